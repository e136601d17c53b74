// locks_select: page scoring (Eq. (1)), per-head page-mass shares, the GQA
// share-average and the forced-page top-(k-2) selection of
// "Locks: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", section 4 ("Score") and Cor. 3.
//
// Two kernels, the second launched as a programmatic dependent of the first:
//
// score_kernel (persistent): the candidate pages of every (sequence b, KV
// head h) "unit" are laid end to end (mc slots per unit) and every CTA takes
// one contiguous, equal range of slots.  Each of its 4 warps owns a
// two-stage shared-memory ring of page-pair slots; lane 0 streams the summary
// records of the warp's next two pages into a slot with 1-D bulk copies, and
// each half-warp (16 lanes) scores one page of the pair:
//   lane l of a half holds dims [4l, 4l+4) and [64+4l, 64+4l+4) of the G
//   group queries and dots them with the centroid and basis rows
//   (a_g = q_g.mu, p_gk = q_g.v_k; packed fp32 pairs along the dims); the
//   G(R+1) partial sums are reduced across the 16 lanes with transposed
//   reductions; the projections go through shared memory to every lane, which
//   forms the reconstructed logits of tokens l, l+16, l+32, l+48 for every
//   head and reduces them by log-sum-exp (transposed max and sum).
// It writes s_hat per (page, head) and, per warp and unit, the running
// (max, sum) log-sum-exp of its s_hat values.
//
// finalize_kernel: CTA (slice, unit) merges the unit's partials into
// log Z_g, forms the averaged shares m_bar_j of its slice of candidates and
// keeps the slice's top-(k-2) (4-pass 8-bit radix select over the share bit
// patterns; ties to the smaller page).  The last slice of the unit (atomic
// ticket, no waiting) merges the slices' winners the same way and writes the
// forced pages and the winners in ascending page order.
#include <mutex>

#include "locks_score.cuh"
#include "locks_topk.cuh"

namespace locks {

namespace {

constexpr int kFinThreads = 256;
constexpr int kFinWarps = kFinThreads / 32;

template <int G>
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const SelectParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  // launched as a programmatic dependent of the score kernel; the decode that
  // follows may begin launching once every CTA here has started
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = blockIdx.y, sl = blockIdx.x;
  const int b = u / p.n_kv_heads;
  const int seq_len = unit_seq_len(p, b);
  const int B = p.page_size;
  if (p.seq_lens[b] > p.max_pages * B && sl == 0 && tid == 0)
    flag_status(p.status, LOCKS_DEV_BAD_SEQ_LEN);
  const int n = (seq_len + B - 1) / B;
  const int n_cand = cand_count(seq_len, B);
  const int nsl = max(1, (n_cand + p.slice - 1) / p.slice);
  if (sl >= nsl) return;
  const int k = p.k, K = k - 2;
  int32_t* out = p.selected + size_t(u) * k;

  __shared__ float s_red[kFinWarps][16][2];
  __shared__ float s_logz[16];
  __shared__ int s_cnt[kFinWarps];
  __shared__ int s_is_last;
  const float* ws_s = p.ws_scores + size_t(u) * p.max_pages * G;
  const int c_lo = sl * p.slice, c_n = min(n_cand, c_lo + p.slice) - c_lo;
  // the register path's score loads go out first: they do not depend on log Z
  float sv_early[8][G];
  const bool early = n > k && K > 0 && K <= 32;
  if (early) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = warp * 256 + 32 * e + lane;
      if (i < c_n) ld_scores<G>(ws_s + size_t(1 + c_lo + i) * G, sv_early[e]);
    }
  }
  // shared memory: keys[cap] pages[cap] | warp winners wk/wp [8][K] | list lk/lp [8K] | hist [8][256]
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  int* pages = reinterpret_cast<int*>(keys + p.fin_cap);
  uint32_t* wk = reinterpret_cast<uint32_t*>(pages + p.fin_cap);
  int* wp = reinterpret_cast<int*>(wk + kFinWarps * K);
  uint32_t* lk = reinterpret_cast<uint32_t*>(wp + kFinWarps * K);
  int* lp = reinterpret_cast<int*>(lk + kFinWarps * K);
  unsigned* hist = reinterpret_cast<unsigned*>(lp + kFinWarps * K) + warp * 256;

  // ---- log Z_g from the unit's partials: block max, then the rescaled sum ----
  {
    const int i_first = int((long(u) * p.mc) / p.per_cta);
    const int i_last = int((long(u + 1) * p.mc - 1) / p.per_cta);
    const int nseg = (i_last - i_first + 1) * 4;
    float m[G], s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) { m[g] = -INFINITY; s[g] = 0.f; }
    for (int sg = tid; sg < nseg; sg += kFinThreads) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float2 v = __ldcg(p.ws_part + (size_t(u) * p.nseg_max + sg) * G + g);
        lse_merge(m[g], s[g], v.x, v.y);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = m[g];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      if (lane == 0) s_red[warp][g][0] = mx;
    }
    __syncthreads();
    float M[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      M[g] = s_red[0][g][0];
      for (int w = 1; w < kFinWarps; ++w) M[g] = fmaxf(M[g], s_red[w][g][0]);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x = (m[g] == -INFINITY) ? 0.f : s[g] * ex2_approx((m[g] - M[g]) * kLog2e);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
      if (lane == 0) s_red[warp][g][1] = x;
    }
    __syncthreads();
    if (tid < G) {
      float ss = 0.f, mt = -INFINITY;
      for (int w = 0; w < kFinWarps; ++w) {
        ss += s_red[w][tid][1];
        mt = fmaxf(mt, s_red[w][tid][0]);
      }
      s_logz[tid] = (ss > 0.f && mt != -INFINITY) ? mt + kLn2 * lg2_approx(ss) : -INFINITY;
    }
    __syncthreads();
  }

  // ---- averaged shares of this slice's candidates ---------------------------
  // warp w owns entries [256w, 256w + 256) of the slice, lane l every 32nd
  const bool select = n > k && K > 0;
  if (early) {
    // ---- register path: sorting networks, no shared-memory passes -------------
    __shared__ unsigned long long s_top[kFinWarps][32];
    __shared__ unsigned long long s_stage[kFinWarps][64];
    unsigned long long v[8];
    {
      float lz2[G];
#pragma unroll
      for (int g = 0; g < G; ++g) lz2[g] = s_logz[g] * kLog2e;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int i = warp * 256 + 32 * e + lane;
        v[e] = 0ull;                                   // below every real candidate
        if (i < c_n) {
          float mb = 0.f;
#pragma unroll
          for (int g = 0; g < G; ++g) mb += ex2_approx(fmaf(sv_early[e][g], kLog2e, -lz2[g]));
          mb *= 1.f / G;
          v[e] = cand_key(__float_as_uint(mb), uint32_t(1 + c_lo + i));
          if (p.page_share) p.page_share[size_t(u) * p.max_pages + 1 + c_lo + i] = mb;
        }
      }
    }
    // warps whose 256 entries lie past the slice's candidates hold nothing
    s_top[warp][lane] = warp * 256 < c_n ? warp_top32_filtered(v, s_stage[warp], lane) : 0ull;
    __syncthreads();
    if (warp == 0) {
      unsigned long long t[kFinWarps];
#pragma unroll
      for (int w = 0; w < kFinWarps; ++w) t[w] = s_top[w][lane];
#pragma unroll
      for (int w = 0; w < kFinWarps; w += 2) t[w] = warp_merge_top32(t[w], t[w + 1], lane);
#pragma unroll
      for (int w = 0; w < kFinWarps; w += 4) t[w] = warp_merge_top32(t[w], t[w + 2], lane);
      t[0] = warp_merge_top32(t[0], t[4], lane);
      if (nsl == 1) {
        warp_emit_pages_ascending(t[0], K, out + 1, lane);
        if (lane == 0) { out[0] = 0; out[k - 1] = n - 1; }
      } else {
        uint2* cand = p.ws_cand + (size_t(u) * p.nslices_max + sl) * p.cand_per_slice;
        cand[lane] = make_uint2(uint32_t(t[0] >> 32), uint32_t(t[0]));
      }
    }
    if (nsl == 1) return;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_is_last = (atomicAdd(p.ws_ticket + u, 1) == nsl - 1);
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    if (warp == 0) {
      unsigned long long acc = 0ull;
      for (int s2 = 0; s2 < nsl; ++s2) {
        const uint2 e = __ldcg(p.ws_cand + (size_t(u) * p.nslices_max + s2) * p.cand_per_slice + lane);
        const unsigned long long x = (static_cast<unsigned long long>(e.x) << 32) | e.y;
        acc = s2 == 0 ? x : warp_merge_top32(acc, x, lane);
      }
      warp_emit_pages_ascending(acc, K, out + 1, lane);
      if (lane == 0) { out[0] = 0; out[k - 1] = n - 1; p.ws_ticket[u] = 0; }
    }
    return;
  }
  {
    float logz[G];
#pragma unroll
    for (int g = 0; g < G; ++g) logz[g] = s_logz[g];
    constexpr int PER = 8;
    for (int base = 0; base < c_n; base += PER * kFinThreads) {
      const int i0 = base + warp * 32 * PER + lane;
      float sv[PER][G];
#pragma unroll
      for (int e = 0; e < PER; ++e)
        if (i0 + 32 * e < c_n) ld_scores<G>(ws_s + size_t(1 + c_lo + i0 + 32 * e) * G, sv[e]);
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const int i = i0 + 32 * e;
        if (i < c_n) {
          float mb = 0.f;
#pragma unroll
          for (int g = 0; g < G; ++g) mb += expf(sv[e][g] - logz[g]);
          mb *= 1.f / G;
          if (select) { keys[i] = __float_as_uint(mb); pages[i] = 1 + c_lo + i; }
          if (p.page_share) p.page_share[size_t(u) * p.max_pages + 1 + c_lo + i] = mb;
        }
      }
    }
  }
  if (!select) {
    if (sl == 0) {
      if (n <= k) {
        for (int t = tid; t < k; t += kFinThreads) out[t] = t < n ? t : -1;
      } else if (tid == 0) {               // k == 2: the forced pages only
        out[0] = 0;
        out[1] = n - 1;
      }
    }
    return;
  }
  __syncthreads();

  // ---- this slice's top-K: per warp over 256 entries, then warp 0 merges ------
  {
    const int w_lo = warp * 256, w_m = max(0, min(c_n - w_lo, 256));
    const int c = warp_topk(keys + w_lo, pages + w_lo, w_m, K, wk + warp * K, wp + warp * K, hist);
    if (lane == 0) s_cnt[warp] = c;
  }
  __syncthreads();
  if (warp == 0) {
    // concatenate the warp winners in warp order (page order is kept)
    int off = 0;
    for (int w = 0; w < kFinWarps; ++w) {
      const int c = s_cnt[w];
      for (int i = lane; i < c; i += 32) { lk[off + i] = wk[w * K + i]; lp[off + i] = wp[w * K + i]; }
      off += c;
    }
    __syncwarp();
    const int got = warp_topk(lk, lp, off, K, wk, wp, hist);
    if (nsl == 1) {
      for (int i = lane; i < K; i += 32) out[1 + i] = wp[i];   // increasing page order
      if (lane == 0) { out[0] = 0; out[k - 1] = n - 1; }
    } else {
      uint2* cand = p.ws_cand + (size_t(u) * p.nslices_max + sl) * p.cand_per_slice;
      for (int i = lane; i < K; i += 32)
        cand[i] = i < got ? make_uint2(wk[i], uint32_t(wp[i])) : make_uint2(0u, 0xffffffffu);
    }
  }
  if (nsl == 1) return;

  // ---- several slices: the last one merges the slices' winners ---------------
  __threadfence();
  __syncthreads();
  if (tid == 0) s_is_last = (atomicAdd(p.ws_ticket + u, 1) == nsl - 1);
  __syncthreads();
  if (!s_is_last) return;
  __threadfence();
  if (warp == 0) {
    // slices in order, each in page order, empty entries (page -1) dropped
    int off = 0;
    for (int s2 = 0; s2 < nsl; ++s2) {
      const uint2* src = p.ws_cand + (size_t(u) * p.nslices_max + s2) * p.cand_per_slice;
      for (int i0 = 0; i0 < K; i0 += 32) {
        const int i = i0 + lane;
        uint2 e = make_uint2(0u, 0xffffffffu);
        if (i < K) e = __ldcg(src + i);
        const bool ok = i < K && e.y != 0xffffffffu;
        const unsigned bal = __ballot_sync(kFull, ok);
        if (ok) {
          const int at = off + __popc(bal & ((1u << lane) - 1));
          keys[at] = e.x;
          pages[at] = int(e.y);
        }
        off += __popc(bal);
      }
    }
    __syncwarp();
    warp_topk(keys, pages, off, K, wk, wp, hist);
    for (int i = lane; i < K; i += 32) out[1 + i] = wp[i];
    if (lane == 0) { out[0] = 0; out[k - 1] = n - 1; p.ws_ticket[u] = 0; }
  }
}

template <int G>
int launch_finalize(const SelectParams& p, int n_slices, cudaStream_t stream) {
  const int K = p.k > 2 ? p.k - 2 : 1;
  const size_t fsmem = size_t(p.fin_cap) * 8 + size_t(kFinWarps) * K * 8 * 2 +
                       size_t(kFinWarps) * 256 * sizeof(unsigned);
  if (fsmem > kMaxDynSmem) return LOCKS_ERR_UNSUPPORTED;
  auto fk = finalize_kernel<G>;
  if (cudaFuncSetAttribute(fk, cudaFuncAttributeMaxDynamicSharedMemorySize, int(fsmem)) !=
      cudaSuccess)
    return LOCKS_ERR_CUDA;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(n_slices, p.units);
  lc.blockDim = dim3(kFinThreads);
  lc.dynamicSmemBytes = fsmem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, fk, p) == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

SelectGeom select_geometry(int units, int max_pages, int G, int k, int ctas_per_sm) {
  SelectGeom g;
  const int K = k > 2 ? k - 2 : 1;
  g.mc = (max_pages > 2 ? max_pages - 2 : 1);
  g.mc += g.mc & 1;                                   // even: page pairs never straddle units
  const long total = long(units) * g.mc;
  // about ctas_per_sm CTAs per SM on 152 SMs, at least 16 slots each, a CTA
  // spanning at most kUnitSlots units, and the slot ids of one CTA in shared
  // memory
  const long ctas = long(ctas_per_sm > 0 ? ctas_per_sm : 2) * 152;
  long per = (total + ctas - 1) / ctas;
  per += per & 1;
  if (per < 16) per = 16;
  if (per > 2048) per = 2048;
  const long cap = long(kUnitSlots - 2) * g.mc;
  if (per > cap) per = cap & ~1L;
  g.per_cta = int(per);
  g.n_score_ctas = int(total > 0 ? (total + per - 1) / per : 1);
  g.nseg_max = ((g.mc + g.per_cta - 1) / g.per_cta + 1) * kSelWarps;
  g.slice = 2048;
  g.nslices_max = (g.mc + g.slice - 1) / g.slice;
  if (g.nslices_max < 1) g.nslices_max = 1;
  g.cand_per_slice = K > 32 ? K : 32;
  g.fin_cap = g.slice > g.nslices_max * K ? g.slice : g.nslices_max * K;
  const size_t U = size_t(units);
  g.off_scores = 0;
  g.off_part = align256(U * max_pages * G * sizeof(float));
  g.off_cand = g.off_part + align256(U * g.nseg_max * G * sizeof(float2));
  g.off_ticket = g.off_cand + align256(U * g.nslices_max * g.cand_per_slice * sizeof(uint2));
  g.total = g.off_ticket + align256(U * sizeof(int32_t));
  return g;
}

int launch_score_b64(const SelectParams& p, int G, int RP, int dtype, int n_ctas,
                     cudaStream_t stream) {
  return launch_score_pb<64>(p, G, RP, dtype, n_ctas, stream);
}

int launch_select(const SelectParams& p, int G, int RP, int dtype, int n_score_ctas,
                  int n_slices, cudaStream_t stream) {
  if (G != 1 && G != 2 && G != 4 && G != 8) return LOCKS_ERR_UNSUPPORTED;
  int rc = p.page_size == 64   ? launch_score_b64(p, G, RP, dtype, n_score_ctas, stream)
           : p.page_size == 16 ? launch_score_b16(p, G, RP, dtype, n_score_ctas, stream)
                               : LOCKS_ERR_UNSUPPORTED;
  if (rc != LOCKS_OK) return rc;
  switch (G) {
    case 1: return launch_finalize<1>(p, n_slices, stream);
    case 2: return launch_finalize<2>(p, n_slices, stream);
    case 4: return launch_finalize<4>(p, n_slices, stream);
    default: return launch_finalize<8>(p, n_slices, stream);
  }
}

}  // namespace locks
