// Selection helpers of the finalize kernel: score loads, block-wide scans and
// the block top-K over a shared-memory list of share bit patterns (a lower
// bound from the per-thread maxima, then a direct ranking of the few keys at
// or above it; a bit-by-bit search of the K-th key when too many are).
// Internal to the library.
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

constexpr int kFinThreads = 256;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kMaxSlice = 2048;              // candidates of one finalize CTA

// Exclusive prefix, in thread order, of x over the block; s_warp holds
// kFinWarps ints and must not be reused before the next block barrier.
__device__ __forceinline__ int block_excl_scan(int x, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int inc = warp_incl_scan(x, lane);
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  int before = 0;
#pragma unroll
  for (int w = 0; w < kFinWarps; ++w) before += w < warp ? s_warp[w] : 0;
  return before + inc - x;
}

// The K-th largest (1 <= K < m) of the keys keys[0..m) in shared memory.
// Returns (T, need): that key, and how many of the keys equal to T are among
// the K largest (at least 1).  A most-significant-bit-first search: with the
// bits above b fixed, the block counts the keys that match them and have bit b
// set; if fewer than the rank still wanted, T has bit b clear and those keys
// all rank above it.  Bit 31 is clear in every key (the keys are non-negative
// floats), so 31 counts decide T, each one warp reduction and one barrier
// (s_cnt: two rows of kFinWarps ints, used alternately).  No histogram: keys
// that crowd into a few values cost nothing extra.
__device__ __forceinline__ uint2 block_radix_select(const uint32_t* keys, int m, int K,
                                                    int (*s_cnt)[kFinWarps]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0u;
  int krem = K;
#pragma unroll 1
  for (int b = 30; b >= 0; --b) {
    const uint32_t hi = ~((2u << b) - 1u);       // the bits above b (fixed so far)
    int c = 0;
    for (int i = tid; i < m; i += kFinThreads) {
      const uint32_t key = keys[i];
      c += ((key & hi) == prefix && (key & (1u << b)) != 0u) ? 1 : 0;
    }
    c = __reduce_add_sync(kFull, c);
    if (lane == 0) s_cnt[b & 1][warp] = c;
    __syncthreads();
    int cnt = 0;
#pragma unroll
    for (int w = 0; w < kFinWarps; ++w) cnt += s_cnt[b & 1][w];
    if (cnt >= krem) prefix |= 1u << b;
    else krem -= cnt;
  }
  return make_uint2(prefix, uint32_t(krem));
}

// Calls put(i, pos) for the entries of the K largest keys -- every key above T
// and the first `need` keys equal to T -- in index order, pos = 0, 1, ...
// Each thread takes a contiguous run of entries; one block scan of the
// packed counts (above T in the high 16 bits, equal in the low) places it.
template <typename F>
__device__ __forceinline__ void block_emit_topk(const uint32_t* keys, int m, uint32_t T, int need,
                                                int* s_warp, F&& put) {
  const int tid = threadIdx.x;
  const int per = (m + kFinThreads - 1) / kFinThreads;
  const int i0 = min(m, tid * per), i1 = min(m, i0 + per);
  int gt = 0, eq = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = keys[i];
    gt += key > T ? 1 : 0;
    eq += key == T ? 1 : 0;
  }
  const int ex = block_excl_scan((gt << 16) | eq, s_warp);
  int ties = ex & 0xffff;
  int pos = (ex >> 16) + min(ties, need);
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = keys[i];
    bool take = key > T;
    if (key == T) {
      take = ties < need;
      ++ties;
    }
    if (take) put(i, pos++);
  }
}

// Rank of key `mine` (at index `me`) among keys[0..m): how many are larger,
// or equal at a smaller index.  A plain loop: this code runs once per step,
// usually from a cold instruction cache, where a short loop beats an
// unrolled one.
__device__ __forceinline__ int rank_in(const uint32_t* keys, int m, uint32_t mine, int me) {
  int r = 0;
  for (int j = 0; j < m; ++j) {
    const uint32_t o = keys[j];
    r += (o > mine || (o == mine && j < me)) ? 1 : 0;
  }
  return r;
}

// Calls put(i, pos) for the K largest (1 <= K < m <= kFinThreads) of the keys
// keys[0..m) -- ordered by key, then by smaller index -- in
// index order: thread i ranks key i against all m keys directly, one scan
// places the winners.  For short lists this beats bounding and compacting
// first.
template <typename F>
__device__ __forceinline__ void block_topk_small(const uint32_t* keys, int m, int K, int* s_warp,
                                                 F&& put) {
  const int tid = threadIdx.x;
  bool win = false;
  if (tid < m) win = rank_in(keys, m, keys[tid], tid) < K;
  const int pos = block_excl_scan(win ? 1 : 0, s_warp);
  if (win) put(tid, pos);
}

constexpr int kSurvCap = 1024;               // survivors the ranking path holds

// Shared-memory scratch of block_topk.
struct alignas(16) TopkScratch {
  uint32_t sk[kSurvCap];                     // survivors: key (16-byte aligned)
  int si[kSurvCap];                          //            index
  uint32_t wj[kFinWarps];                    // per warp: its j-th largest thread maximum
  int scan[6][kFinWarps];
};

// Calls put(i, pos) for the K largest (1 <= K < m, K <= kFinThreads) of the
// keys keys[0..m) in shared memory -- ordered by key, then by smaller index --
// in index order, pos = 0, 1, ...
//
// Each thread takes a contiguous run of the keys.  With j = ceil(K / 8), the
// smallest over the 8 warps of each warp's j-th largest thread maximum is a
// lower bound of the K-th largest key (8j >= K keys reach it); only keys at
// or above it survive, usually a few dozen.  The survivors,
// compacted in index order, are ranked against one another directly and the
// winners placed by one block scan -- a handful of barriers in all.  When
// more survive than kSurvCap holds (many equal keys), the bit-by-bit search
// of the K-th key decides instead.
template <typename F>
__device__ __forceinline__ void block_topk(const uint32_t* keys, int m, int K, TopkScratch& S,
                                           F&& put) {
  const int tid = threadIdx.x;
  const int per = (m + kFinThreads - 1) / kFinThreads;
  const int i0 = min(m, tid * per), i1 = min(m, i0 + per);
  uint32_t mx = 0u;                            // a thread without keys: 0, which
  for (int i = i0; i < i1; ++i) mx = max(mx, keys[i]);   // only lets every key through
  {
    // rank of this lane's maximum in its warp (ties: lower lane first)
    const int lane = tid & 31, j = (K + kFinWarps - 1) / kFinWarps;
    int r = 0;
#pragma unroll 4
    for (int d = 1; d < 32; ++d) {
      const int o_lane = (lane + d) & 31;
      const uint32_t o = __shfl_sync(kFull, mx, o_lane);
      r += (o > mx || (o == mx && o_lane < lane)) ? 1 : 0;
    }
    if (r == j - 1) S.wj[tid >> 5] = mx;
  }
  __syncthreads();
  uint32_t lb = S.wj[0];
#pragma unroll
  for (int w = 1; w < kFinWarps; ++w) lb = min(lb, S.wj[w]);
  int c = 0;
  for (int i = i0; i < i1; ++i) c += keys[i] >= lb ? 1 : 0;
  int n_surv = 0;
  {
    const int lane = tid & 31, warp = tid >> 5;
    const int inc = warp_incl_scan(c, lane);
    if (lane == 31) S.scan[0][warp] = inc;
    __syncthreads();
    int before = 0;
#pragma unroll
    for (int w = 0; w < kFinWarps; ++w) {
      const int x = S.scan[0][w];
      before += w < warp ? x : 0;
      n_surv += x;
    }
    if (n_surv <= kSurvCap) {
      int at = before + inc - c;
      for (int i = i0; i < i1; ++i)
        if (keys[i] >= lb) { S.sk[at] = keys[i]; S.si[at] = i; ++at; }
    }
  }
  if (n_surv > kSurvCap) {
    const uint2 sel = block_radix_select(keys, m, K, S.scan + 1);
    block_emit_topk(keys, m, sel.x, int(sel.y), S.scan[3], put);
    return;
  }
  __syncthreads();
  // rank every survivor; winners are those of rank < K.  Thread t takes a
  // contiguous run of survivors so that one scan places the winners in order.
  const int ps = (n_surv + kFinThreads - 1) / kFinThreads;
  const int j0 = min(n_surv, tid * ps), j1 = min(n_surv, j0 + ps);
  uint32_t win = 0u;                           // bit q: survivor j0 + q wins (ps <= 4)
  int nw = 0;
  for (int j = j0; j < j1; ++j) {
    if (rank_in(S.sk, n_surv, S.sk[j], j) < K) { win |= 1u << (j - j0); ++nw; }
  }
  const int pos0 = block_excl_scan(nw, S.scan[4]);
  int pos = pos0;
  for (int j = j0; j < j1; ++j)
    if (win & (1u << (j - j0))) put(S.si[j], pos++);
}

}  // namespace
}  // namespace locks
