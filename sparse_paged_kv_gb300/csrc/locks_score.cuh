// Page scoring of locks_select (Eq. (1) of "Locks: Page-Local Compact Key
// Summaries for Efficient Long-Context Decoding", section 4 "Score"): the
// score kernel (each CTA streams one contiguous range of candidate pages),
// templated on the page size B (64 or 16).  Included by one translation unit
// per page size; internal to the library.
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


// floats of one half-warp's projection buffer: G*R padded to 16 bytes; for
// the quantised record half a warp's [2][17][8] pair buffer
template <int G, int RP, typename T>
__host__ __device__ constexpr int pbuf_stride() {
  return std::is_same_v<T, I4Rec> ? 17 * 8 : (G * RP + 3) / 4 * 4;
}

// q . w over this lane's 8 dims: packed fp32 pairs along the dims, then one add
__device__ __forceinline__ float dot8(const float4& qa, const float4& qb, const float4& wa,
                                      const float4& wb) {
  float2 acc = fmul2(make_float2(qa.x, qa.y), make_float2(wa.x, wa.y));
  acc = ffma2(make_float2(qa.z, qa.w), make_float2(wa.z, wa.w), acc);
  acc = ffma2(make_float2(qb.x, qb.y), make_float2(wb.x, wb.y), acc);
  acc = ffma2(make_float2(qb.z, qb.w), make_float2(wb.z, wb.w), acc);
  return acc.x + acc.y;
}

// ---- quantised record: tensor-core scorer -----------------------------------
// The int4 basis and the int8 centroid and coefficients are exact small
// integers in f16, so both contractions of Eq. (1) run as f16 mma with f32
// accumulators: the projection P = V^T q (basis rows against the group's
// queries) and the logits C P (coefficient rows against P).  The scales are
// applied to the f32 results: per basis column to P, per row to the logits.

// D += A . B, f16 operands, f32 accumulators (m16n8k16 and m16n8k8)
__device__ __forceinline__ void mma_f16_k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// The biased 4-bit codes in bits 0-3 and 16-19 of w as the f16 pair
// (code - 8): the nibble is placed in the low mantissa bits of 1024 (0x6400),
// whose unit in the last place is 1, and 1032 is taken off.  nib2_hi_f16
// does the same for bits 4-7 and 20-23 without a shift: under 64 (0x5400)
// the unit in the last place is 1/16, so mantissa bits 4-7 count whole units
// and 72 is taken off.  Every step is exact.
__device__ __forceinline__ uint32_t nib2_f16(uint32_t w) {
  const uint32_t x = (w & 0x000F000Fu) | 0x64006400u;
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x64086408u));
  return r;
}
__device__ __forceinline__ uint32_t nib2_hi_f16(uint32_t w) {
  const uint32_t x = (w & 0x00F000F0u) | 0x54005400u;
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x54805480u));
  return r;
}
// Two biased 8-bit codes of w (bytes picked by `sel`, 0x4140 for bytes 0 and
// 1, 0x4342 for bytes 2 and 3) as the f16 pair (code - 128), the same way.
__device__ __forceinline__ uint32_t byte2_f16(uint32_t w, uint32_t sel) {
  const uint32_t x = __byte_perm(w, 0x64u, sel);
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x64806480u));
  return r;
}
__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 f16x2_to_f2(uint32_t h) {
  float lo, hi;
  asm("{.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
  return make_float2(lo, hi);
}
// (v0, v1) as an f16 pair hi plus the f16 pair lo of what hi misses, so that
// hi + lo carries about 22 bits of each value
__device__ __forceinline__ void split_f16(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  hi = f16x2(v0, v1);
  const float2 h = f16x2_to_f2(hi);
  lo = f16x2(v0 - h.x, v1 - h.y);
}

// The group's queries of one unit as the B operand of the projection: for
// k-step s (dims 16s..16s+15) lane 4g+t holds head g's dims 16s+2t, +1 in
// b[s][0] and 16s+2t+8, +9 in b[s][1] (zero for g >= G), scaled by the power
// of two 2^-e that puts max|q| in [512, 1024): exact for every bf16 value in
// f16's normal range, and the projection sums stay far inside f16's range.
struct QFrag {
  uint32_t b[8][2];
  float pw;                                   // 2^e
};
template <int G>
__device__ __forceinline__ void load_qfrag(QFrag& f, const __nv_bfloat16* qh, int lane) {
  const int g = lane >> 2, t = lane & 3;
  uint32_t raw[8][2];
  float mx = 0.f;
#pragma unroll
  for (int s = 0; s < 8; ++s)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      raw[s][h] = g < G ? *reinterpret_cast<const uint32_t*>(qh + g * kHeadDim + 16 * s + 2 * t +
                                                             8 * h)
                        : 0u;
      mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(raw[s][h] << 16)),
                           fabsf(__uint_as_float(raw[s][h] & 0xffff0000u))));
    }
  mx = group_max<32>(mx);
  const int E = max(int((__float_as_uint(mx) >> 23) & 0xff) - 127, -117);
  const float down = __uint_as_float(uint32_t(136 - E) << 23);   // 2^(9 - E)
  f.pw = __uint_as_float(uint32_t(118 + E) << 23);               // 2^(E - 9)
#pragma unroll
  for (int s = 0; s < 8; ++s)
#pragma unroll
    for (int h = 0; h < 2; ++h)
      f.b[s][h] = f16x2(__uint_as_float(raw[s][h] << 16) * down,
                        __uint_as_float(raw[s][h] & 0xffff0000u) * down);
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  unsigned long long ra, rb, rd;
  ra = *reinterpret_cast<unsigned long long*>(&a);
  rb = *reinterpret_cast<unsigned long long*>(&b);
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  return *reinterpret_cast<float2*>(&rd);
}
__device__ __forceinline__ float2 shfl_xor2(float2 v, int o) {
  return make_float2(__shfl_xor_sync(kFull, v.x, o), __shfl_xor_sync(kFull, v.y, o));
}

// Scores the two quantised page summaries of a slot pair (records r0 and
// r0 + rec_bytes) with the whole warp; pb is the warp's [2][17][8] pair
// buffer.  Returns, in lane 16 * p + hl, s_hat of page p and head hl / (16/G).
//
// Projection (per page, 8 k-steps of m16n8k16): A rows g are the basis codes
// of column g (R <= 8; for R = 16 rows g + 8 hold column g + 8 and the
// centroid takes 8 more mma), B is the query fragment, D[k][n] = P~_k of head
// n.  For R <= 8 the centroid rides in A rows 8..15: row 8 + s carries the
// centroid's dims of k-step s only, so summing D rows 8..15 gives mu . q~.
// Logits (per page or, for G <= 4, both pages in one accumulator with page p
// in columns 4p..4p+3 through a block-diagonal B): A = coefficient codes of 16
// tokens, B = the scaled projections as hi + lo f16 pairs.
template <int G, int RP, int PB>
__device__ __forceinline__ float score_pair_i4(const unsigned char* r0, uint32_t rec_bytes,
                                               const QFrag& qf, float* pb, float scale,
                                               float scale_log2, int lane) {
  constexpr bool kPack = G <= 4;              // both pages in one logits accumulator
  constexpr int NSET = kPack ? 1 : 2;
  constexpr int MT = PB / 16;                 // 16-token tiles of a page
  constexpr int KK = i4_kk(RP);
  constexpr int kPS = 17 * 8;                 // floats of a page's part of pb
  const int g = lane >> 2, t = lane & 3;

  // ---- projection and centroid term of both pages (two mma chains) ---------
  const uint4 pad = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
  uint4 w0[2], w1[2];                         // basis codes of column g (and g + 8)
  uint32_t m01[2], m89[2];                    // centroid codes of k-step g
  float d[2][4], dm[2][4];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const unsigned char* rb = r0 + p * rec_bytes;
    const uint4* vq = reinterpret_cast<const uint4*>(rb + i4_vq(RP));
    w0[p] = g < RP ? vq[g * 4 + t] : pad;                // code 8 is the value 0
    w1[p] = pad;
    if constexpr (RP > 8) w1[p] = vq[(g + 8) * 4 + t];
    const uint32_t mw = reinterpret_cast<const uint32_t*>(rb + i4_mq(RP))[lane];
    m01[p] = byte2_f16(mw, 0x4140u);
    m89[p] = byte2_f16(mw, 0x4342u);
#pragma unroll
    for (int e = 0; e < 4; ++e) d[p][e] = dm[p][e] = 0.f;
  }
  auto word = [](const uint4& w, int j) { return j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w; };
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t keep = g == s ? 0xffffffffu : 0u;     // the centroid's k-step s row
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const uint32_t wa = word(w0[p], s >> 1) >> (8 * (s & 1));
      const uint32_t a0 = nib2_f16(wa), a2 = nib2_hi_f16(wa);
      if constexpr (RP <= 8) {
        mma_f16_k16(d[p], a0, m01[p] & keep, a2, m89[p] & keep, qf.b[s][0], qf.b[s][1]);
      } else {
        const uint32_t wb = word(w1[p], s >> 1) >> (8 * (s & 1));
        mma_f16_k16(d[p], a0, nib2_f16(wb), a2, nib2_hi_f16(wb), qf.b[s][0], qf.b[s][1]);
        mma_f16_k16(dm[p], m01[p] & keep, 0u, m89[p] & keep, 0u, qf.b[s][0], qf.b[s][1]);
      }
    }
  }
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    // P_k (times 2^-e) of heads 2t, 2t+1 for k = g (and g + 8)
    const float* hdr = reinterpret_cast<const float*>(r0 + p * rec_bytes);
    float* pp = pb + p * kPS;
    const float vs0 = g < RP ? hdr[g] : 0.f;
    *reinterpret_cast<float2*>(pp + g * 8 + 2 * t) = make_float2(d[p][0] * vs0, d[p][1] * vs0);
    float c0 = d[p][2], c1 = d[p][3];
    if constexpr (RP > 8) {
      const float vs1 = hdr[g + 8];
      *reinterpret_cast<float2*>(pp + (g + 8) * 8 + 2 * t) =
          make_float2(d[p][2] * vs1, d[p][3] * vs1);
      c0 = dm[p][0];
      c1 = dm[p][1];
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      c0 += __shfl_xor_sync(kFull, c0, o);
      c1 += __shfl_xor_sync(kFull, c1, o);
    }
    if (g == 0) {
      const float ms = hdr[RP];
      *reinterpret_cast<float2*>(pp + 128 + 2 * t) = make_float2(c0 * ms, c1 * ms);
    }
  }
  __syncwarp();

  // ---- logits: B operands from the pair buffer ------------------------------
  // lane 4g+t supplies column g: P_k of k = 2t, 2t+1 (and 2t+8, 2t+9)
  uint32_t bh[2][2], bl[2][2];                // [page][k half]
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const float* src = kPack ? pb + (g >> 2) * kPS + (g & 3) : pb + p * kPS + g;
    if (kPack && p == 1) {                    // packed: one read serves the lane's own page
      bh[1][0] = bh[0][0]; bl[1][0] = bl[0][0]; bh[1][1] = bh[0][1]; bl[1][1] = bl[0][1];
      continue;
    }
    split_f16(src[(2 * t) * 8], src[(2 * t + 1) * 8], bh[p][0], bl[p][0]);
    bh[p][1] = bl[p][1] = 0u;
    if constexpr (RP > 8) split_f16(src[(2 * t + 8) * 8], src[(2 * t + 9) * 8], bh[p][1], bl[p][1]);
  }
  float acc[NSET][MT][4];
#pragma unroll
  for (int d = 0; d < NSET; ++d)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[d][m][0] = acc[d][m][1] = acc[d][m][2] = acc[d][m][3] = 0.f;
  const uint32_t* cq0 = reinterpret_cast<const uint32_t*>(r0 + i4_cq(RP));
  const uint32_t* cq1 = reinterpret_cast<const uint32_t*>(r0 + rec_bytes + i4_cq(RP));
  const int pg = g >> 2;                      // packed: the page of the lane's B column
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    if constexpr (kPack && RP <= 8) {
      // k 0..7: page 0's coefficients (columns 0..3), k 8..15: page 1's (4..7)
      const uint32_t w0 = cq0[m * 32 + lane], w1 = cq1[m * 32 + lane];
      const uint32_t a0 = byte2_f16(w0, 0x4140u), a1 = byte2_f16(w0, 0x4342u);
      const uint32_t a2 = byte2_f16(w1, 0x4140u), a3 = byte2_f16(w1, 0x4342u);
      const uint32_t h0 = pg == 0 ? bh[0][0] : 0u, h1 = pg == 1 ? bh[0][0] : 0u;
      const uint32_t l0 = pg == 0 ? bl[0][0] : 0u, l1 = pg == 1 ? bl[0][0] : 0u;
      mma_f16_k16(acc[0][m], a0, a1, a2, a3, h0, h1);
      mma_f16_k16(acc[0][m], a0, a1, a2, a3, l0, l1);
    } else {
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const uint32_t* cq = p == 0 ? cq0 : cq1;
        float (&ac)[4] = acc[kPack ? 0 : p][m];
        const uint32_t w0 = cq[(m * KK) * 32 + lane];
        const uint32_t a0 = byte2_f16(w0, 0x4140u), a1 = byte2_f16(w0, 0x4342u);
        if constexpr (RP <= 8) {
          mma_f16_k8(ac, a0, a1, bh[p][0]);
          mma_f16_k8(ac, a0, a1, bl[p][0]);
        } else {
          const uint32_t w1 = cq[(m * KK + 1) * 32 + lane];
          const uint32_t a2 = byte2_f16(w1, 0x4140u), a3 = byte2_f16(w1, 0x4342u);
          const bool own = !kPack || pg == p;
          mma_f16_k16(ac, a0, a1, a2, a3, own ? bh[p][0] : 0u, own ? bh[p][1] : 0u);
          mma_f16_k16(ac, a0, a1, a2, a3, own ? bl[p][0] : 0u, own ? bl[p][1] : 0u);
        }
      }
    }
  }

  // ---- log-sum-exp per (page, head) over the page's tokens ------------------
  // accumulator d, lane 4g+t: tokens 16m+g (elements 0, 1) and 16m+g+8 (2, 3)
  // of columns 2t, 2t+1; packed, column c is head c % 4 of page c / 4
  const float cu = qf.pw * scale_log2;
  const float2 cu2 = make_float2(cu, cu);
  float res[NSET][2];
#pragma unroll
  for (int d = 0; d < NSET; ++d) {
    const int page = kPack ? (t >> 1) : d;
    const unsigned char* rb = r0 + page * rec_bytes;
    const float* cs = reinterpret_cast<const float*>(rb + i4_cscale(RP, PB));
    float2 z[MT][2];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float s0 = cs[16 * m + g], s1 = cs[16 * m + g + 8];
      z[m][0] = fmul2(make_float2(acc[d][m][0], acc[d][m][1]), make_float2(s0, s0));
      z[m][1] = fmul2(make_float2(acc[d][m][2], acc[d][m][3]), make_float2(s1, s1));
      mx0 = fmaxf(mx0, fmaxf(z[m][0].x, z[m][1].x));
      mx1 = fmaxf(mx1, fmaxf(z[m][0].y, z[m][1].y));
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
    }
    const float mc0 = mx0 * cu, mc1 = mx1 * cu;
    const float2 nmc = make_float2(-mc0, -mc1);
    float2 e = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float2 x = ffma2(z[m][r], cu2, nmc);
        e = fadd2(e, make_float2(ex2_approx(x.x), ex2_approx(x.y)));
      }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) e = fadd2(e, shfl_xor2(e, o));
    const float e0 = e.x, e1 = e.y;
    const float2 a = *reinterpret_cast<const float2*>(pb + page * kPS + 128 +
                                                      (kPack ? 2 * (t & 1) : 2 * t));
    const float sa = scale * qf.pw;
    res[d][0] = fmaf(sa, a.x, kLn2 * (mc0 + lg2_approx(e0)));
    res[d][1] = fmaf(sa, a.y, kLn2 * (mc1 + lg2_approx(e1)));
  }
  __syncwarp();                               // pb is rewritten by the next pair

  // ---- to the head lanes: lane 16p + hl takes page p, head hl / (16/G) ------
  const int page = lane >> 4, head = (lane & 15) / (kHalf / G);
  float v0 = res[0][0], v1 = res[0][1];
  if constexpr (!kPack) {
    v0 = page ? res[NSET - 1][0] : res[0][0];
    v1 = page ? res[NSET - 1][1] : res[0][1];
  }
  const int src = kPack ? 2 * page + (head >> 1) : (lane & 16) + (head >> 1);
  const float r0v = __shfl_sync(kFull, v0, src), r1v = __shfl_sync(kFull, v1, src);
  return (head & 1) ? r1v : r0v;
}

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

  float pv[NP];
  float av[G];
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
  TransposeReduce<NP, kHalf / 2>::run(pv, lane);
  TransposeReduce<G, kHalf / 2>::run(av, lane);
  // lane hl holds p values [(hl / (16/SP)) * VP, +VP) and a of head hl / LG
  if ((hl & (kHalf / SP - 1)) == 0) {
#pragma unroll
    for (int e = 0; e < VP; ++e) pbuf[(hl / (kHalf / SP)) * VP + e] = pv[e];
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
      const float4 c = ld4(rec + rec_w_elems(RP) + (cc * PB + i) * 4);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        acc[g] = ffma2(make_float2(pr[g][cc].x, pr[g][cc].y), make_float2(c.x, c.y), acc[g]);
        acc[g] = ffma2(make_float2(pr[g][cc].z, pr[g][cc].w), make_float2(c.z, c.w), acc[g]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) x[g][t] = acc[g].x + acc[g].y;
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
__global__ void __launch_bounds__(kSelThreads, (!std::is_same_v<T, I4Rec> &&
                                                 (G >= 8 || G * RP >= 64 || sizeof(T) == 4))
                                                    ? 2
                                                    : 4)
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
  constexpr bool kI4 = std::is_same_v<T, I4Rec>;
  float* pbuf = pbuf_all + (warp * 2 + (kI4 ? 0 : half)) * pbuf_stride<G, RP, T>();
  float2* upart = reinterpret_cast<float2*>(pbuf_all + kSelWarps * 2 * pbuf_stride<G, RP, T>());
  // per slot: x = record index (block * n_kv_heads + h) if valid, -1 invalid
  // (flagged), -2 no such candidate; y = (unit - u_lo) << 24 | page index j
  int2* s_slot = reinterpret_cast<int2*>(upart + kSelWarps * kUnitSlots * G);   // [n_f]

  uint64_t* mybar = bars + warp * STAGES;
  unsigned char* myring = ring + size_t(warp) * STAGES * 2 * rec_bytes;
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(mybar + s, 1);
    mbar_fence_init();
  }
  // launched as a programmatic dependent of the previous kernel in the stream
  // (in a decode loop, the append of the step's token): everything below
  // reads what that kernel may write
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int t = tid; t < n_f; t += kSelThreads) {
    const long f = f_lo + t;
    const int u = int(f / p.mc), idx = int(f % p.mc);
    const int b = u / p.n_kv_heads, h = u % p.n_kv_heads;
    int v = -2;
    if (idx < cand_count(unit_seq_len(p, b), PB)) {
      const int blk = p.block_table[size_t(b) * p.max_pages + 1 + idx];
      v = (blk >= 0 && blk < p.num_blocks) ? blk * p.n_kv_heads + h : -1;
      if (v == -1) flag_status(p.status, LOCKS_DEV_BAD_BLOCK_ID);
    }
    s_slot[t] = make_int2(v, ((u - u_lo) << 24) | (1 + idx));
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
    const int b0 = s_slot[t0].x, b1 = s_slot[t0 + 1].x;
    const uint32_t bytes = uint32_t(rec_bytes) * ((b0 >= 0) + (b1 >= 0));
    if (bytes) {
      mbar_arrive_expect_tx(mybar + s, bytes);
      const uint64_t pol = l2_evict_first();
      if (b0 >= 0)
        bulk_g2s_hint(myring + size_t(2 * s) * rec_bytes, sum_base + size_t(b0) * rec_bytes,
                      uint32_t(rec_bytes), mybar + s, pol);
      if (b1 >= 0)
        bulk_g2s_hint(myring + size_t(2 * s + 1) * rec_bytes, sum_base + size_t(b1) * rec_bytes,
                      uint32_t(rec_bytes), mybar + s, pol);
    } else {
      mbar_arrive(mybar + s);
    }
  };
  // Quantised records: each warp asks for its first page pair alone and for
  // the second once the first has landed.  Every warp of the grid asks at
  // once, so halving that opening burst lands each first pair sooner, and the
  // tensor-core scoring, which takes about as long as the copies, starts
  // sooner (llama32k select 27.8 -> 27.0 us).  Float records keep both in
  // the burst: their scoring is short and the stream alone bounds them.
  if (lane == 0)
    for (int i = 0; i < min(kI4 ? 1 : STAGES, my_count); ++i) issue(i);

  const int my_head = hl / LG;
  const bool head_lane = (hl % LG) == 0;
  int cur_u = -1, cur_b = 0, cur_h = 0;
  float zm = -INFINITY, zs = 0.f;              // running LSE of the current unit (head lanes)
  float4 qa[G], qb[G];
  QFrag qf;
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
    const int2 slot = s_slot[t0 + half];       // both slots of a pair share the unit
    const int u = u_lo + (slot.y >> 24);
    if (u != cur_u) {                          // warp-uniform
      flush();
      cur_u = u;
      cur_b = u / p.n_kv_heads;
      cur_h = u - cur_b * p.n_kv_heads;
      const int b = cur_b, h = cur_h;
      if constexpr (kI4) {
        load_qfrag<G>(qf, p.q + (size_t(b) * (p.n_kv_heads * G) + h * G) * kHeadDim, lane);
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const __nv_bfloat16* qg =
              p.q + (size_t(b) * (p.n_kv_heads * G) + h * G + g) * kHeadDim;
          qa[g] = bf16x4_to_f4(*reinterpret_cast<const uint2*>(qg + 4 * hl));
          qb[g] = bf16x4_to_f4(*reinterpret_cast<const uint2*>(qg + 64 + 4 * hl));
        }
      }
    }
    if (!__all_sync(kFull, mbar_wait_bounded(mybar + s, (i / STAGES) & 1))) {
      if (lane == 0) flag_status(p.status, LOCKS_DEV_WAIT_TIMEOUT);
      aborted = true;
      done = i;
      break;
    }
    if constexpr (kI4) {
      if (i == 0 && lane == 0 && 1 < my_count) issue(1);
    }
    float shat;
    if constexpr (kI4)
      shat = score_pair_i4<G, RP, PB>(myring + size_t(2 * s) * rec_bytes, uint32_t(rec_bytes), qf,
                                      pbuf, p.scale, p.scale_log2, lane);
    else
      shat = score_page16<G, RP, T, PB>(
          reinterpret_cast<const T*>(myring + size_t(2 * s + half) * rec_bytes), qa, qb, pbuf, hl,
          p.scale, p.scale_log2);
    if (head_lane && slot.x != -2) {
      const int j = slot.y & 0xffffff;
      const float v = slot.x >= 0 ? shat : -INFINITY;
      p.ws_scores[(size_t(u) * p.max_pages + j) * G + my_head] = v;
      if (p.page_lse)
        p.page_lse[(size_t(cur_b) * (p.n_kv_heads * G) + cur_h * G + my_head) * p.max_pages + j] =
            v;
      if (slot.x >= 0) lse_merge(zm, zs, v, 1.f);
    }
    __syncwarp();
    if (lane == 0 && i + STAGES < my_count) issue(i + STAGES);
  }
  if (aborted) {
    // let the copies still in flight land before the CTA can exit
    const int in_flight_end =
        (kI4 && done == 0) ? min(my_count, 1) : min(my_count, done + STAGES);
    for (int i = done; i < in_flight_end; ++i)
      mbar_wait_bounded(mybar + (i % STAGES), (i / STAGES) & 1);
  }
  flush();

  // the dependent grid (the finalize kernel) may start launching; it waits for
  // this grid's completion before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();

  // merge the warps' partials of every unit this CTA touched and write one
  // (max, sum) pair per (CTA, unit, head): the finalize then reads a quarter
  // as many segments
  for (int t = tid; t < (u_hi - u_lo + 1) * G; t += kSelThreads) {
    const int g = t % G, us = t / G;
    const int u = u_lo + us;
    float m = -INFINITY, s = 0.f;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      const float2 v = upart[(w * kUnitSlots + us) * G + g];
      lse_merge(m, s, v.x, v.y);
    }
    const int i_first = int((long(u) * p.mc) / p.per_cta);
    p.ws_part[(size_t(u) * p.nseg_max + (int(blockIdx.x) - i_first)) * G + g] = make_float2(m, s);
  }
}

template <int G, int RP, typename T, int PB>
int launch_score_t(const SelectParams& p, int n_ctas, cudaStream_t stream) {
  // ring depth: two page pairs per warp.  Deeper rings (tried for the small
  // quantised record) only make the opening burst of copies longer: every
  // warp's first pair then lands later, and the tensor-core scoring, which
  // takes about as long as the copies, starts later.
  constexpr int STAGES = 2;
  const size_t smem = size_t(kSelWarps) * STAGES * 2 * p.rec_bytes +
                      kSelWarps * STAGES * sizeof(uint64_t) +
                      kSelWarps * 2 * pbuf_stride<G, RP, T>() * sizeof(float) +
                      kSelWarps * kUnitSlots * G * sizeof(float2) + size_t(p.per_cta) * sizeof(int2);
  if (smem > kMaxDynSmem) return LOCKS_ERR_UNSUPPORTED;
  auto sk = score_kernel<G, RP, T, STAGES, PB>;
  if (cudaFuncSetAttribute(sk, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return LOCKS_ERR_CUDA;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(n_ctas);
  lc.blockDim = dim3(kSelThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, sk, p) == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
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
