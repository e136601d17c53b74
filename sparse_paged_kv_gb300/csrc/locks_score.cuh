// Page scoring of locks_select (Eq. (1) of "Locks: Page-Local Compact Key
// Summaries for Efficient Long-Context Decoding", section 4 "Score"): the
// persistent score kernel, templated on the page size B (64 or 16).  Included
// by one translation unit per page size; internal to the library.
#pragma once

#include <type_traits>

#include "locks_common.cuh"
#include "locks_internal.h"

namespace locks {

constexpr int kSelWarps = 4;
constexpr int kSelThreads = kSelWarps * 32;
constexpr int kHalf = 16;                    // lanes per page
constexpr int kUnitSlots = 16;               // units one score CTA may touch

// sequence length clamped to the block table; candidates are the complete
// pages other than page 0 and page n-1
__device__ __forceinline__ int unit_seq_len(const SelectParams& p, int b) {
  int t = p.seq_lens[b];
  if (t > p.max_pages * p.page_size) t = p.max_pages * p.page_size;
  return t < 0 ? 0 : t;
}
__device__ __forceinline__ int cand_count(int seq_len, int B) {
  const int n = (seq_len + B - 1) / B;
  const int hi = min(n - 1, seq_len / B);
  return max(0, hi - 1);
}

namespace {


// floats of one half-warp's projection buffer (G*R, padded to 16 bytes)
template <int G, int RP>
__host__ __device__ constexpr int pbuf_stride() { return (G * RP + 3) / 4 * 4; }

// q . w over this lane's 8 dims: packed fp32 pairs along the dims, then one add
__device__ __forceinline__ float dot8(const float4& qa, const float4& qb, const float4& wa,
                                      const float4& wb) {
  float2 acc = fmul2(make_float2(qa.x, qa.y), make_float2(wa.x, wa.y));
  acc = ffma2(make_float2(qa.z, qa.w), make_float2(wa.z, wa.w), acc);
  acc = ffma2(make_float2(qb.x, qb.y), make_float2(wb.x, wb.y), acc);
  acc = ffma2(make_float2(qb.z, qb.w), make_float2(wb.z, wb.w), acc);
  return acc.x + acc.y;
}

// Four biased codes (the bytes of w) as floats minus their bias: each byte is
// placed in the mantissa of 2^23 (exact) and 2^23 + bias is subtracted.
__device__ __forceinline__ float4 biased_bytes_f4(uint32_t w, float bias_plus_2p23) {
  return make_float4(__int_as_float(__byte_perm(w, 0x4B000000u, 0x7540)) - bias_plus_2p23,
                     __int_as_float(__byte_perm(w, 0x4B000000u, 0x7541)) - bias_plus_2p23,
                     __int_as_float(__byte_perm(w, 0x4B000000u, 0x7542)) - bias_plus_2p23,
                     __int_as_float(__byte_perm(w, 0x4B000000u, 0x7543)) - bias_plus_2p23);
}
constexpr float kI4Off = 8388616.f;     // 2^23 + 8   (int4 codes stored + 8)
constexpr float kI8Off = 8388736.f;     // 2^23 + 128 (int8 codes stored + 128)

// Scores one page summary `rec` in each half-warp (lane hl = lane % 16 of the
// half).  Returns s_hat of head hl / (16/G) (identical across that head's lanes).
template <int G, int RP, typename T, int PB>
__device__ __forceinline__ float score_page16(const T* __restrict__ rec, const float4 (&qa)[G],
                                              const float4 (&qb)[G], float* pbuf, int hl,
                                              float scale, float scale_log2) {
  constexpr int NP = G * RP;                   // basis projections p_{g,k}
  constexpr int SP = NP < kHalf ? NP : kHalf;
  constexpr int VP = NP / SP;                  // values a lane holds after the reduction
  constexpr int LG = kHalf / G;                // lanes per head after the G-value reductions
  const int lane = threadIdx.x & 31;

  constexpr bool kI4 = std::is_same_v<T, I4Rec>;
  const unsigned char* rb = reinterpret_cast<const unsigned char*>(rec);
  float pv[NP];
  float av[G];
  if constexpr (kI4) {
    // quantised record: codes -> floats, dot, then the group scales after the
    // reductions (a = mscale * q.codes(mu), p_k = vscale[k] * q.codes(v_k))
    const uint2 mw = reinterpret_cast<const uint2*>(rb + i4_mq(RP))[hl];
    const float4 wa = biased_bytes_f4(mw.x, kI8Off), wb = biased_bytes_f4(mw.y, kI8Off);
#pragma unroll
    for (int g = 0; g < G; ++g) av[g] = dot8(qa[g], qb[g], wa, wb);
    const uint32_t* vq = reinterpret_cast<const uint32_t*>(rb + i4_vq(RP));
#pragma unroll
    for (int k = 0; k < RP; ++k) {
      const uint32_t w = vq[k * 16 + hl];
      const float4 va = biased_bytes_f4(w & 0x0F0F0F0Fu, kI4Off);
      const float4 vb = biased_bytes_f4((w >> 4) & 0x0F0F0F0Fu, kI4Off);
#pragma unroll
      for (int g = 0; g < G; ++g) pv[g * RP + k] = dot8(qa[g], qb[g], va, vb);
    }
  } else {
    {
      const float4 wa = ld4(rec + 4 * hl), wb = ld4(rec + 64 + 4 * hl);   // centroid
#pragma unroll
      for (int g = 0; g < G; ++g) av[g] = dot8(qa[g], qb[g], wa, wb);
    }
#pragma unroll
    for (int k = 0; k < RP; ++k) {
      const float4 wa = ld4(rec + (1 + k) * kHeadDim + 4 * hl);
      const float4 wb = ld4(rec + (1 + k) * kHeadDim + 64 + 4 * hl);
#pragma unroll
      for (int g = 0; g < G; ++g) pv[g * RP + k] = dot8(qa[g], qb[g], wa, wb);
    }
  }
  TransposeReduce<NP, kHalf / 2>::run(pv, lane);
  TransposeReduce<G, kHalf / 2>::run(av, lane);
  // lane hl holds p values [(hl / (16/SP)) * VP, +VP) and a of head hl / LG
  if constexpr (kI4) av[0] *= reinterpret_cast<const float*>(rb)[RP];
  if ((hl & (kHalf / SP - 1)) == 0) {
#pragma unroll
    for (int e = 0; e < VP; ++e) {
      const int idx = (hl / (kHalf / SP)) * VP + e;
      if constexpr (kI4) pbuf[idx] = pv[e] * reinterpret_cast<const float*>(rb)[idx % RP];
      else pbuf[idx] = pv[e];
    }
  }
  __syncwarp();

  // reconstructed logits (before the 1/sqrt(d) scale) of tokens hl + 16t
  constexpr int TPL = PB / kHalf;              // tokens per lane (4 or 1)
  float4 pr[G][RP / 4];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int cc = 0; cc < RP / 4; ++cc)
      pr[g][cc] = *reinterpret_cast<const float4*>(pbuf + g * RP + cc * 4);
  float x[G][TPL];
#pragma unroll
  for (int t = 0; t < TPL; ++t) {
    float2 acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = make_float2(0.f, 0.f);
    const int i = hl + kHalf * t;
#pragma unroll
    for (int cc = 0; cc < RP / 4; ++cc) {
      float4 c;
      if constexpr (kI4)
        c = biased_bytes_f4(reinterpret_cast<const uint32_t*>(rb + i4_cq(RP) + i * RP)[cc], kI8Off);
      else
        c = ld4(rec + rec_w_elems(RP) + (cc * PB + i) * 4);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        acc[g] = ffma2(make_float2(pr[g][cc].x, pr[g][cc].y), make_float2(c.x, c.y), acc[g]);
        acc[g] = ffma2(make_float2(pr[g][cc].z, pr[g][cc].w), make_float2(c.z, c.w), acc[g]);
      }
    }
    float row = 1.f;                            // the row's scale (quantised record)
    if constexpr (kI4) row = reinterpret_cast<const float*>(rb + i4_cscale(RP, PB))[i];
#pragma unroll
    for (int g = 0; g < G; ++g) x[g][t] = (acc[g].x + acc[g].y) * row;
  }
  // log-sum-exp per head: transposed max, broadcast, exponentials, transposed sum
  float mx[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    mx[g] = x[g][0];
#pragma unroll
    for (int t = 1; t < TPL; ++t) mx[g] = fmaxf(mx[g], x[g][t]);
  }
  TransposeMax<G, kHalf / 2>::run(mx, lane);   // lane holds the max of head hl / LG
  const float my_max = mx[0];
  float ev[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float m = __shfl_sync(kFull, my_max, g * LG, kHalf);
    const float mc = m * scale_log2;
    float e = 0.f;
#pragma unroll
    for (int t = 0; t < TPL; ++t) e += ex2_approx(fmaf(x[g][t], scale_log2, -mc));
    ev[g] = e;
  }
  TransposeReduce<G, kHalf / 2>::run(ev, lane);   // lane holds the sum of head hl / LG
  __syncwarp();                                   // pbuf is rewritten by the next page
  return scale * (av[0] + my_max) + kLn2 * lg2_approx(ev[0]);
}


template <int G, int RP, typename T, int STAGES, int PB>
__global__ void __launch_bounds__(kSelThreads, (G >= 8 || G * RP >= 64 || sizeof(T) == 4) ? 2 : 4)
    score_kernel(const SelectParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int half = lane >> 4, hl = lane & 15;
  constexpr int LG = kHalf / G;
  const long total = long(p.units) * p.mc;
  const long f_lo = long(blockIdx.x) * p.per_cta;
  const long f_hi = min(total, f_lo + p.per_cta);
  if (f_lo >= f_hi) return;
  const int n_f = int(f_hi - f_lo);              // even
  const int u_lo = int(f_lo / p.mc);
  const int u_hi = int((f_hi - 1) / p.mc);       // u_hi - u_lo < kUnitSlots

  // ---- shared memory ------------------------------------------------------
  const size_t rec_bytes = p.rec_bytes;
  unsigned char* ring = smem;
  const size_t ring_bytes = size_t(kSelWarps) * STAGES * 2 * rec_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_bytes);
  float* pbuf_all = reinterpret_cast<float*>(bars + kSelWarps * STAGES);
  float* pbuf = pbuf_all + (warp * 2 + half) * pbuf_stride<G, RP>();
  float2* upart = reinterpret_cast<float2*>(pbuf_all + kSelWarps * 2 * pbuf_stride<G, RP>());
  int* s_blk = reinterpret_cast<int*>(upart + kSelWarps * kUnitSlots * G);   // [n_f]

  uint64_t* mybar = bars + warp * STAGES;
  unsigned char* myring = ring + size_t(warp) * STAGES * 2 * rec_bytes;
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(mybar + s, 1);
    mbar_fence_init();
  }
  // block id of every slot: >= 0 valid, -1 invalid (flagged), -2 no such candidate
  for (int t = tid; t < n_f; t += kSelThreads) {
    const long f = f_lo + t;
    const int u = int(f / p.mc), idx = int(f % p.mc);
    const int b = u / p.n_kv_heads;
    int v = -2;
    if (idx < cand_count(unit_seq_len(p, b), PB)) {
      const int blk = p.block_table[size_t(b) * p.max_pages + 1 + idx];
      v = (blk >= 0 && blk < p.num_blocks) ? blk : -1;
      if (v == -1) flag_status(p.status, LOCKS_DEV_BAD_BLOCK_ID);
    }
    s_blk[t] = v;
  }
  for (int t = tid; t < kSelWarps * kUnitSlots * G; t += kSelThreads)
    upart[t] = make_float2(-INFINITY, 0.f);
  __syncthreads();

  // warp w scores the slot pairs (2q, 2q+1), q = w, w+4, ...; both slots of a
  // pair belong to the same unit (mc and the range start are even)
  const int n_pairs = n_f / 2;
  const int my_count = (n_pairs - warp + kSelWarps - 1) / kSelWarps;   // may be <= 0
  const unsigned char* sum_base = static_cast<const unsigned char*>(p.summaries);
  auto issue = [&](int i) {
    const int s = i % STAGES;
    const int t0 = 2 * (i * kSelWarps + warp);
    const int h = int((f_lo + t0) / p.mc) % p.n_kv_heads;
    const int b0 = s_blk[t0], b1 = s_blk[t0 + 1];
    const uint32_t bytes = uint32_t(rec_bytes) * ((b0 >= 0) + (b1 >= 0));
    if (bytes) {
      mbar_arrive_expect_tx(mybar + s, bytes);
      if (b0 >= 0)
        bulk_g2s(myring + size_t(2 * s) * rec_bytes,
                 sum_base + (size_t(b0) * p.n_kv_heads + h) * rec_bytes, uint32_t(rec_bytes),
                 mybar + s);
      if (b1 >= 0)
        bulk_g2s(myring + size_t(2 * s + 1) * rec_bytes,
                 sum_base + (size_t(b1) * p.n_kv_heads + h) * rec_bytes, uint32_t(rec_bytes),
                 mybar + s);
    } else {
      mbar_arrive(mybar + s);
    }
  };
  if (lane == 0)
    for (int i = 0; i < min(STAGES, my_count); ++i) issue(i);

  const int my_head = hl / LG;
  const bool head_lane = (hl % LG) == 0;
  int cur_u = -1;
  float zm = -INFINITY, zs = 0.f;              // running LSE of the current unit (head lanes)
  float4 qa[G], qb[G];
  auto flush = [&]() {                         // merge the halves, keep in the unit slot
    const float m2 = __shfl_xor_sync(kFull, zm, kHalf), s2 = __shfl_xor_sync(kFull, zs, kHalf);
    lse_merge(zm, zs, m2, s2);
    if (cur_u >= 0 && half == 0 && head_lane)
      upart[(warp * kUnitSlots + (cur_u - u_lo)) * G + my_head] = make_float2(zm, zs);
    zm = -INFINITY;
    zs = 0.f;
  };
  bool aborted = false;
  int done = 0;
  for (int i = 0; i < my_count; ++i) {
    const int s = i % STAGES;
    const int t0 = 2 * (i * kSelWarps + warp);
    const int u = int((f_lo + t0) / p.mc);
    if (u != cur_u) {                          // warp-uniform
      flush();
      cur_u = u;
      const int b = u / p.n_kv_heads, h = u % p.n_kv_heads;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const __nv_bfloat16* qg = p.q + (size_t(b) * (p.n_kv_heads * G) + h * G + g) * kHeadDim;
        qa[g] = bf16x4_to_f4(*reinterpret_cast<const uint2*>(qg + 4 * hl));
        qb[g] = bf16x4_to_f4(*reinterpret_cast<const uint2*>(qg + 64 + 4 * hl));
      }
    }
    if (!__all_sync(kFull, mbar_wait_bounded(mybar + s, (i / STAGES) & 1))) {
      if (lane == 0) flag_status(p.status, LOCKS_DEV_WAIT_TIMEOUT);
      aborted = true;
      done = i;
      break;
    }
    const int t = t0 + half;
    const int blk = s_blk[t];
    const float shat = score_page16<G, RP, T, PB>(
        reinterpret_cast<const T*>(myring + size_t(2 * s + half) * rec_bytes), qa, qb, pbuf, hl,
        p.scale, p.scale_log2);
    if (head_lane && blk != -2) {
      const int j = 1 + int((f_lo + t) % p.mc);
      const int b = u / p.n_kv_heads, h = u % p.n_kv_heads;
      const float v = blk >= 0 ? shat : -INFINITY;
      p.ws_scores[(size_t(u) * p.max_pages + j) * G + my_head] = v;
      if (p.page_lse)
        p.page_lse[(size_t(b) * (p.n_kv_heads * G) + h * G + my_head) * p.max_pages + j] = v;
      if (blk >= 0) lse_merge(zm, zs, v, 1.f);
    }
    __syncwarp();
    if (lane == 0 && i + STAGES < my_count) issue(i + STAGES);
  }
  if (aborted) {
    // let the copies still in flight land before the CTA can exit
    for (int i = done; i < min(my_count, done + STAGES); ++i)
      mbar_wait_bounded(mybar + (i % STAGES), (i / STAGES) & 1);
  }
  flush();

  // the dependent grid (the finalize kernel) may start launching; it waits for
  // this grid's completion before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();

  // write the per-(warp, unit) partials of every unit this CTA touched
  for (int t = tid; t < kSelWarps * (u_hi - u_lo + 1) * G; t += kSelThreads) {
    const int g = t % G, w = (t / G) % kSelWarps, us = t / (G * kSelWarps);
    const int u = u_lo + us;
    const int i_first = int((long(u) * p.mc) / p.per_cta);
    const int seg = (int(blockIdx.x) - i_first) * kSelWarps + w;
    p.ws_part[(size_t(u) * p.nseg_max + seg) * G + g] = upart[(w * kUnitSlots + us) * G + g];
  }
}

template <int G, int RP, typename T, int PB>
int launch_score_t(const SelectParams& p, int n_ctas, cudaStream_t stream) {
  // ring depth: enough record bytes in flight per warp to cover the memory
  // latency (a quantised record is about a fifth of a float one)
  constexpr int STAGES = std::is_same_v<T, I4Rec> ? 4 : 2;
  const size_t smem = size_t(kSelWarps) * STAGES * 2 * p.rec_bytes +
                      kSelWarps * STAGES * sizeof(uint64_t) +
                      kSelWarps * 2 * pbuf_stride<G, RP>() * sizeof(float) +
                      kSelWarps * kUnitSlots * G * sizeof(float2) + size_t(p.per_cta) * sizeof(int);
  if (smem > kMaxDynSmem) return LOCKS_ERR_UNSUPPORTED;
  auto sk = score_kernel<G, RP, T, STAGES, PB>;
  if (cudaFuncSetAttribute(sk, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return LOCKS_ERR_CUDA;
  sk<<<n_ctas, kSelThreads, smem, stream>>>(p);
  return cudaPeekAtLastError() == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
}

template <typename T, int PB>
int score_dispatch(const SelectParams& p, int G, int RP, int n_ctas, cudaStream_t s) {
#define LOCKS_SCORE_CASE(GG, RR) \
  if (G == GG && RP == RR) return launch_score_t<GG, RR, T, PB>(p, n_ctas, s);
  LOCKS_SCORE_CASE(1, 4) LOCKS_SCORE_CASE(1, 8) LOCKS_SCORE_CASE(1, 16)
  LOCKS_SCORE_CASE(2, 4) LOCKS_SCORE_CASE(2, 8) LOCKS_SCORE_CASE(2, 16)
  LOCKS_SCORE_CASE(4, 4) LOCKS_SCORE_CASE(4, 8) LOCKS_SCORE_CASE(4, 16)
  LOCKS_SCORE_CASE(8, 4) LOCKS_SCORE_CASE(8, 8) LOCKS_SCORE_CASE(8, 16)
#undef LOCKS_SCORE_CASE
  return LOCKS_ERR_UNSUPPORTED;
}

}  // namespace

// The score kernel for page size PB (instantiated once per page size).
template <int PB>
int launch_score_pb(const SelectParams& p, int G, int RP, int dtype, int n_ctas,
                    cudaStream_t stream) {
  if (dtype == LOCKS_SUMMARY_F32) return score_dispatch<float, PB>(p, G, RP, n_ctas, stream);
  if (dtype == LOCKS_SUMMARY_I4) return score_dispatch<I4Rec, PB>(p, G, RP, n_ctas, stream);
  return score_dispatch<__nv_bfloat16, PB>(p, G, RP, n_ctas, stream);
}

}  // namespace locks
