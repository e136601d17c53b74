// Device helpers shared by the Locks kernels (sm_103a).
//
// * 1-D bulk copies global -> shared (cp.async.bulk) completing on an mbarrier
//   with a transaction count;
// * bounded mbarrier waits: every wait gives up after a wall-clock limit,
//   records LOCKS_DEV_WAIT_TIMEOUT and lets the caller skip the work;
// * warp "transpose" reductions: N per-lane partial sums are reduced across
//   the lanes of a warp (or of an aligned lane group) with N-1 shuffles in
//   total, each lane ending with the full sums of its share of the N values.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/locks.h"

namespace locks {

constexpr int kHeadDim = 128;
constexpr unsigned kFull = 0xffffffffu;
// A bounded wait on a copy gives up after this many nanoseconds.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__host__ __device__ constexpr int rank_cap(int r) { return r <= 4 ? 4 : (r <= 8 ? 8 : 16); }

// Record geometry (element counts); see the record description in locks.h.
__host__ __device__ constexpr int rec_w_elems(int rp) { return (rp + 1) * kHeadDim; }
__host__ __device__ constexpr int rec_elems(int rp, int B) { return (rp + 1) * kHeadDim + rp * B; }

// Quantised record (LOCKS_SUMMARY_I4) byte offsets; see the layout in locks.h.
__host__ __device__ constexpr int i4_hdr(int rp) { return ((rp + 1) * 4 + 15) / 16 * 16; }
__host__ __device__ constexpr int i4_vq(int rp) { return i4_hdr(rp); }
__host__ __device__ constexpr int i4_mq(int rp) { return i4_hdr(rp) + 64 * rp; }
__host__ __device__ constexpr int i4_cq(int rp) { return i4_mq(rp) + 128; }
__host__ __device__ constexpr int i4_kk(int rp) { return (rp + 7) / 8; }
__host__ __device__ constexpr int i4_cscale(int rp, int B) { return i4_cq(rp) + 8 * B * i4_kk(rp); }
__host__ __device__ constexpr int i4_bytes(int rp, int B) { return i4_cscale(rp, B) + 4 * B; }

// Tag type of the quantised record in the kernels' templates.
struct I4Rec {};

// ---------------------------------------------------------------------------
// status words
// ---------------------------------------------------------------------------
__device__ __forceinline__ void flag_status(int32_t* status, int32_t bits) {
  if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------
// mbarrier + bulk copy
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar` to complete; false if the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Copy `bytes` (multiple of 16, both addresses 16-byte aligned) from global to
// shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data a step reads exactly once (summary records, selected and
// dense K/V pages): evicted first, so that what the step's later kernels use
// again -- their code, the score workspace, block tables, queries -- stays in
// L2 while hundreds of MB stream through it.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy for the source lines
__device__ __forceinline__ void bulk_g2s_hint(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float4 bf16x4_to_f4(uint2 w) {
  return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
}

__device__ __forceinline__ float ld_elem(const float* p) { return *p; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// four consecutive elements (16 B of float / 8 B of bf16) from shared memory
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  return bf16x4_to_f4(*reinterpret_cast<const uint2*>(p));
}

__device__ __forceinline__ void st_elem(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// ---------------------------------------------------------------------------
// fast base-2 exponent / logarithm (the PTX approximate instructions)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// packed fp32 FMA (two lanes of fp32 per instruction on sm_100+)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ra, rb, rc, rd;
  ra = *reinterpret_cast<unsigned long long*>(&a);
  rb = *reinterpret_cast<unsigned long long*>(&b);
  rc = *reinterpret_cast<unsigned long long*>(&c);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return *reinterpret_cast<float2*>(&rd);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  unsigned long long ra, rb, rd;
  ra = *reinterpret_cast<unsigned long long*>(&a);
  rb = *reinterpret_cast<unsigned long long*>(&b);
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  return *reinterpret_cast<float2*>(&rd);
}

// ---------------------------------------------------------------------------
// Transposed warp reduction.
//
// Every lane of an aligned group of WIDTH lanes (a power of two <= 32) holds
// N partial sums v[0..N) (N a power of two).  After the call, with
// S = min(N, WIDTH), lane l of the group holds in v[0 .. N/S) the group-wide
// sums of the values with indices  (l % WIDTH) / (WIDTH / S) * (N / S) + e.
// It costs N/2 + N/4 + ... shuffles while N halves, then one butterfly
// shuffle per remaining lane bit.
// ---------------------------------------------------------------------------
template <int N, int OFF>
struct TransposeReduce {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (OFF >= 1) {
      if constexpr (N > 1) {
        constexpr int H = N / 2;
        const bool upper = (lane & OFF) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float send = upper ? v[i] : v[i + H];
          const float keep = upper ? v[i + H] : v[i];
          v[i] = keep + __shfl_xor_sync(kFull, send, OFF);
        }
        TransposeReduce<H, OFF / 2>::run(v, lane);
      } else {
        v[0] += __shfl_xor_sync(kFull, v[0], OFF);
        TransposeReduce<1, OFF / 2>::run(v, lane);
      }
    }
  }
};

// Transposed max: as TransposeReduce with max in place of +.
template <int N, int OFF>
struct TransposeMax {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (OFF >= 1) {
      if constexpr (N > 1) {
        constexpr int H = N / 2;
        const bool upper = (lane & OFF) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float send = upper ? v[i] : v[i + H];
          const float keep = upper ? v[i + H] : v[i];
          v[i] = fmaxf(keep, __shfl_xor_sync(kFull, send, OFF));
        }
        TransposeMax<H, OFF / 2>::run(v, lane);
      } else {
        v[0] = fmaxf(v[0], __shfl_xor_sync(kFull, v[0], OFF));
        TransposeMax<1, OFF / 2>::run(v, lane);
      }
    }
  }
};

// Plain butterfly max / sum over an aligned group of WIDTH lanes.
template <int WIDTH>
__device__ __forceinline__ float group_max(float x) {
#pragma unroll
  for (int o = WIDTH / 2; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
  return x;
}
template <int WIDTH>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = WIDTH / 2; o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

// Online log-sum-exp state merge: (m, s) represents s * exp(m) (natural log).
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  // branch-free: with both sides empty (max -inf) the sum stays 0
  const float M = fmaxf(m, m2);
  const float Mr = M == -INFINITY ? 0.f : M;
  s = s * __expf(m - Mr) + s2 * __expf(m2 - Mr);
  m = M;
}

}  // namespace locks
