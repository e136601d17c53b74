// Warp-level selection helpers of the finalize kernel: candidate keys (share
// bits above the inverted page id), register sorting networks over 32 lanes,
// and a radix top-K over a shared-memory list.  Internal to the library.
#pragma once

#include "locks_common.cuh"

namespace locks {
namespace {

// G scores of one page from the workspace (16-byte loads where G allows)
template <int G>
__device__ __forceinline__ void ld_scores(const float* src, float (&v)[G]) {
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int g = 0; g < G; g += 4) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(src + g));
      v[g] = x.x; v[g + 1] = x.y; v[g + 2] = x.z; v[g + 3] = x.w;
    }
  } else if constexpr (G == 2) {
    const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
    v[0] = x.x; v[1] = x.y;
  } else {
    v[0] = __ldcg(src);
  }
}

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// ---------------------------------------------------------------------------
// register sorting networks over 32 lanes (64-bit keys, descending)
// ---------------------------------------------------------------------------
// Composite key of a candidate: share bits above the inverted page id, so a
// larger key is a larger share and, between equal shares, a smaller page.
__device__ __forceinline__ unsigned long long cand_key(uint32_t share_bits, uint32_t page) {
  return (static_cast<unsigned long long>(share_bits) << 32) | (0xffffffffu - page);
}
__device__ __forceinline__ uint32_t key_page(unsigned long long k) {
  return 0xffffffffu - static_cast<uint32_t>(k);
}

__device__ __forceinline__ unsigned long long shfl_xor64(unsigned long long v, int m) {
  return __shfl_xor_sync(kFull, v, m);
}

// Bitonic sort of one value per lane across the warp, descending in lane order.
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned long long o = shfl_xor64(v, j);
      const bool lower = (lane & j) == 0, first_half = (lane & k) == 0 || k == 32;
      v = (lower == first_half) ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// Given a bitonic sequence across the lanes, sort it descending.
__device__ __forceinline__ unsigned long long warp_bitonic_merge_desc(unsigned long long v,
                                                                     int lane) {
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const unsigned long long o = shfl_xor64(v, j);
    v = ((lane & j) == 0) ? (v > o ? v : o) : (v < o ? v : o);
  }
  return v;
}

// Top 32 of two descending lane-ordered lists, descending.
__device__ __forceinline__ unsigned long long warp_merge_top32(unsigned long long a,
                                                              unsigned long long b, int lane) {
  const unsigned long long br = __shfl_sync(kFull, b, 31 - lane);
  return warp_bitonic_merge_desc(a > br ? a : br, lane);
}

// Sorts each of the 8 per-lane columns and merges them: returns the warp's
// top 32 of its 256 keys, descending in lane order.
__device__ __forceinline__ unsigned long long warp_top32_of_256(unsigned long long (&v)[8],
                                                               int lane) {
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = warp_sort_desc(v[e], lane);
#pragma unroll
  for (int e = 0; e < 8; e += 2) v[e] = warp_merge_top32(v[e], v[e + 1], lane);
#pragma unroll
  for (int e = 0; e < 8; e += 4) v[e] = warp_merge_top32(v[e], v[e + 2], lane);
  return warp_merge_top32(v[0], v[4], lane);
}

// The warp's top 32 of its 256 keys, first discarding every key below the
// smallest of the 32 lane maxima (at least 32 keys reach it, so the top 32 all
// do); the survivors -- usually a few dozen -- are compacted through `stage`
// (64 entries of shared memory) and sorted as two 32-lists.  More than 64
// survivors fall back to sorting all 256.
__device__ __forceinline__ unsigned long long warp_top32_filtered(unsigned long long (&v)[8],
                                                                 unsigned long long* stage,
                                                                 int lane) {
  unsigned long long mx = v[0];
#pragma unroll
  for (int e = 1; e < 8; ++e) mx = v[e] > mx ? v[e] : mx;
  unsigned long long thr = mx;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const unsigned long long x = shfl_xor64(thr, o);
    thr = x < thr ? x : thr;
  }
  int mine = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) mine += v[e] >= thr;
  const int before = warp_incl_scan(mine, lane) - mine;
  const int total = __shfl_sync(kFull, before + mine, 31);
  if (total > 64) return warp_top32_of_256(v, lane);
  stage[lane] = 0ull;
  stage[32 + lane] = 0ull;
  __syncwarp();
  int at = before;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (v[e] >= thr) stage[at++] = v[e];
  __syncwarp();
  const unsigned long long a = warp_sort_desc(stage[lane], lane);
  const unsigned long long b = warp_sort_desc(stage[32 + lane], lane);
  __syncwarp();
  return warp_merge_top32(a, b, lane);
}

// Writes the first K (<= 32) keys of a descending list as pages in increasing
// page order to out[0..K).
__device__ __forceinline__ void warp_emit_pages_ascending(unsigned long long top, int K,
                                                          int32_t* out, int lane) {
  // sort the chosen pages ascending: key = inverted page (descending sort),
  // lanes beyond K get the smallest key
  unsigned long long pk = lane < K ? static_cast<unsigned long long>(0xffffffffu - key_page(top))
                                   : 0ull;
  pk = warp_sort_desc(pk, lane);
  if (lane < K) out[lane] = int32_t(0xffffffffu - static_cast<uint32_t>(pk));
}

// ---------------------------------------------------------------------------
// warp-level top-K over a list kept in increasing page order
// ---------------------------------------------------------------------------
// Chooses the K largest keys of list[0, m) (shared memory, entries in
// increasing page order) with one warp: a 4-pass 8-bit radix select of the
// K-th largest key in a private 256-bin histogram, then the entries above it
// and, among the entries equal to it, the earliest (smaller pages).  The
// chosen entries are written in list order -- still increasing page order --
// to out_keys / out_pages; returns their number, min(K, m).
__device__ int warp_topk(const uint32_t* keys, const int* pages, int m, int K, uint32_t* out_keys,
                         int* out_pages, unsigned* hist) {
  const int lane = threadIdx.x & 31;
  if (m <= K) {
    for (int i = lane; i < m; i += 32) { out_keys[i] = keys[i]; out_pages[i] = pages[i]; }
    __syncwarp();
    return m;
  }
  // lane l looks at entries l, l + 32, l + 64, ... (conflict-free shared loads)
  uint32_t prefix = 0, mask = 0;
  int kleft = K;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
#pragma unroll
    for (int e = 0; e < 8; ++e) hist[e * 32 + lane] = 0;
    __syncwarp();
    for (int i0 = 0; i0 < m; i0 += 32) {
      // one atomic per distinct bin per round (keys crowd into a few bins)
      const int i = i0 + lane;
      uint32_t bin = 256u;                     // not counted
      if (i < m) {
        const uint32_t k = keys[i];
        if ((k & mask) == prefix) bin = (k >> shift) & 255u;
      }
      const unsigned peers = __match_any_sync(kFull, bin);
      if (bin < 256u && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], unsigned(__popc(peers)));
    }
    __syncwarp();
    // lane l owns bins [8*(31-l), 8*(31-l)+8): lane 0 the highest
    unsigned cnt[8], tot = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      cnt[e] = hist[8 * (31 - lane) + 7 - e];
      tot += cnt[e];
    }
    const int incl = warp_incl_scan(int(tot), lane);
    const int first = __ffs(__ballot_sync(kFull, incl >= kleft)) - 1;
    int digit = 0, above = 0;
    if (lane == first) {
      int acc = incl - int(tot);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (acc + int(cnt[e]) >= kleft) { digit = 8 * (31 - lane) + 7 - e; above = acc; break; }
        acc += cnt[e];
      }
    }
    digit = __shfl_sync(kFull, digit, first);
    above = __shfl_sync(kFull, above, first);
    prefix |= uint32_t(digit) << shift;
    mask |= 255u << shift;
    kleft -= above;
    __syncwarp();
  }
  const uint32_t thr = prefix;
  const int need = kleft;                     // entries equal to thr to take
  // collect in list order, 32 entries per round: ballots give the positions
  const unsigned lt = (1u << lane) - 1;
  int pos = 0, eq_seen = 0;
  for (int i0 = 0; i0 < m; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t k = i < m ? keys[i] : 0u;
    const bool eq = i < m && k == thr;
    const unsigned eq_bal = __ballot_sync(kFull, eq);
    const bool take = (i < m && k > thr) || (eq && eq_seen + __popc(eq_bal & lt) < need);
    const unsigned tb = __ballot_sync(kFull, take);
    if (take) {
      const int at = pos + __popc(tb & lt);
      out_keys[at] = k;
      out_pages[at] = pages[i];
    }
    pos += __popc(tb);
    eq_seen += __popc(eq_bal);
  }
  __syncwarp();
  return K;
}

}  // namespace
}  // namespace locks
