// locks_select: page scoring (Eq. (1)), per-head page-mass shares, the GQA
// share-average and the forced-page top-(k-2) selection of
// "Locks: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", section 4 ("Score") and Cor. 3.
//
// Two kernels, the second launched as a programmatic dependent of the first
// (and the sparse decode as one of the second):
//
// score_kernel: the candidate pages of every (sequence b, KV
// head h) "unit" are laid end to end (mc slots per unit) and every CTA takes
// one contiguous, equal range of slots.  Each of its 4 warps owns a
// shared-memory ring of page-pair slots; lane 0 streams the summary records of
// the warp's next two pages into a slot with 1-D bulk copies.  For float and
// bf16 records each half-warp (16 lanes) scores one page of the pair:
//   lane l of a half holds dims [4l, 4l+4) and [64+4l, 64+4l+4) of the G
//   group queries and dots them with the centroid and basis rows
//   (a_g = q_g.mu, p_gk = q_g.v_k; packed fp32 pairs along the dims); the
//   G(R+1) partial sums are reduced across the 16 lanes with transposed
//   reductions; the projections go through shared memory to every lane, which
//   forms the reconstructed logits of tokens l, l+16, l+32, l+48 for every
//   head and reduces them by log-sum-exp (transposed max and sum).
// For the quantised record the whole warp scores the pair with f16 mma (see
// score_pair_i4).  The kernel writes s_hat per (page, head) and, per CTA and
// unit, the (max, sum) log-sum-exp of its s_hat values (its warps' running
// pairs merged in the CTA).
//
// finalize_kernel: CTA (slice, unit) merges the unit's partials into log Z_g
// (each warp by itself), forms the averaged shares m_bar_j of its slice of up
// to 2048 candidates and finds the slice's top-(k-2) (block_topk: a per-warp
// order statistic of the per-thread maxima bounds the answer from below, the
// few shares at or above it are ranked against one another; between equal
// shares the smaller page wins); one block scan writes the winners in page
// order.  A unit of 2 to 8 slices is one thread-block cluster whose CTAs merge
// their winners through distributed shared memory; with more slices the last
// one to finish (atomic ticket, no waiting) selects among the slices' winners.
// Either way the forced pages and the winners are written in ascending page
// order.
//
// The score kernel itself is launched as a programmatic dependent of whatever
// precedes it on the stream, and waits for it before reading anything.
#include <mutex>

#include "locks_score.cuh"
#include "locks_topk.cuh"

namespace locks {

namespace {

// distributed shared memory (the unit's slices as one thread-block cluster)
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ uint2 ld_cluster_u2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
// every thread of every CTA of the cluster; shared-memory writes before it are
// visible to the cluster's loads after it
__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release;\n"
      "barrier.cluster.wait.acquire;" ::: "memory");
}

// CL: the unit's slices form one thread-block cluster (2 to 8 slices) and
// merge their winners through distributed shared memory; otherwise the last
// slice to finish (atomic ticket) merges them from global memory.
template <int G, bool CL>
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const SelectParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  // launched as a programmatic dependent of the score kernel: what it reads
  // before griddepcontrol.wait (the sequence lengths) was complete before the
  // score kernel began; the decode that follows may begin launching once
  // every CTA here has started
  const int tid = threadIdx.x, lane = tid & 31;
  const int u = blockIdx.y, sl = blockIdx.x;
  const int b = u / p.n_kv_heads;
  const int seq_len = unit_seq_len(p, b);
  const int B = p.page_size;
  if (p.seq_lens[b] > p.max_pages * B && sl == 0 && tid == 0)
    flag_status(p.status, LOCKS_DEV_BAD_SEQ_LEN);
  const int n = (seq_len + B - 1) / B;
  const int n_cand = cand_count(seq_len, B);
  const int nsl = max(1, (n_cand + p.slice - 1) / p.slice);
  // shared memory: keys[fin_cap] | pages[fin_cap]
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  int* pages = reinterpret_cast<int*>(keys + p.fin_cap);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int k = p.k, K = k - 2;
  int32_t* out = p.selected + size_t(u) * k;
  const bool select = n > k && K > 0;

  __shared__ TopkScratch ts;
  __shared__ int s_is_last;
  __shared__ uint2 s_win[256];               // clustered merge: this slice's winners
  __shared__ int s_flag[256];
  __shared__ int s_ng, s_off;
  // ---- clustered merge (every CTA of the cluster, n_own winners here) -------
  // Each slice copies all slices' winners (in slice order, so page order) into
  // its own shared memory and ranks its own against them, several threads to
  // a winner; those of rank < K are selected.  A winner's place in the output
  // is the number of selected winners of the slices before it plus its place
  // among its own slice's, so the slices exchange their counts once more.
  // Three cluster barriers: winners written, counts written, counts read.
  auto cluster_merge = [&](int n_own) {
    cluster_barrier();
    int x = 0;
    if (n_own > 0) {                         // uniform in the CTA
      const int m_all = (nsl - 1) * K + min(K, n_cand - (nsl - 1) * p.slice);
      const uint32_t base = smem_u32(s_win);
      for (int i = tid; i < m_all; i += kFinThreads) {
        const int s2 = i / K, e2 = i - s2 * K;
        const uint2 e = ld_cluster_u2(cluster_addr(base + 8u * uint32_t(e2), s2));
        keys[i] = e.x;
        pages[i] = int(e.y);
      }
      __syncthreads();
      const int tpc = n_own <= 32 ? 8 : n_own <= 64 ? 4 : n_own <= 128 ? 2 : 1;
      const int c = tid / tpc, q = tid - c * tpc;
      int r = 0;
      if (c < n_own) {
        const int ge = sl * K + c;
        const uint32_t mine = keys[ge];
        for (int j = q; j < m_all; j += tpc) {
          const uint32_t o = keys[j];
          r += (o > mine || (o == mine && j < ge)) ? 1 : 0;
        }
      }
      for (int o = tpc >> 1; o >= 1; o >>= 1) r += __shfl_xor_sync(kFull, r, o);
      if (c < n_own && q == 0) s_flag[c] = r < K ? 1 : 0;
      __syncthreads();
      x = tid < n_own ? s_flag[tid] : 0;
    }
    const int pos = block_excl_scan(x, ts.scan[0]);
    if (tid == kFinThreads - 1) s_ng = pos + x;
    cluster_barrier();
    if (tid < 32) {
      int v = lane < sl ? ld_cluster_s32(cluster_addr(smem_u32(&s_ng), lane)) : 0;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
      if (lane == 0) s_off = v;
    }
    __syncthreads();
    if (x) out[1 + s_off + pos] = pages[sl * K + tid];
    if (sl == 0 && tid == 0) { out[0] = 0; out[k - 1] = n - 1; }
    cluster_barrier();
  };
  if (sl >= nsl) {
    // in a cluster the slices past the unit's candidates still meet at its
    // barriers (the condition is uniform in the cluster: one unit)
    if constexpr (CL) {
      if (select && nsl > 1) cluster_merge(0);
    }
    return;
  }
  const float* ws_s = p.ws_scores + size_t(u) * p.max_pages * G;
  const int c_lo = sl * p.slice, c_n = min(n_cand, c_lo + p.slice) - c_lo;   // <= slice
  // the slice's scores go out first: they do not depend on log Z
  constexpr int kPer = kMaxSlice / kFinThreads;
  float sv[kPer][G];
  if (select) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i = kFinThreads * e + tid;
      if (i < c_n) ld_scores<G>(ws_s + size_t(1 + c_lo + i) * G, sv[e]);
    }
  }

  // ---- log Z_g from the unit's partials ---------------------------------------
  // Up to 128 segments: every warp merges them itself, so no block barrier
  // separates log Z from the shares.  More (long sequences): the block shares
  // the loads -- one round of them -- and combines the warps' results through
  // shared memory.  Either way each lane merges its segments, then the warp
  // takes the largest max, rescales every lane's sum to it once and adds.
  float lz[G];
  {
    const int i_first = int((long(u) * p.mc) / p.per_cta);
    const int i_last = int((long(u + 1) * p.mc - 1) / p.per_cta);
    const int nseg = i_last - i_first + 1;    // one partial per score CTA
    const bool wide = nseg > 128;
    const int stride = wide ? kFinThreads : 32, first = wide ? tid : lane;
    float m[G], s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) { m[g] = -INFINITY; s[g] = 0.f; }
    // four segments per thread in flight at once, then merged
    for (int sg0 = 0; sg0 < nseg; sg0 += 4 * stride) {
      float2 v[4][G];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int sg = sg0 + stride * r + first;
#pragma unroll
        for (int g = 0; g < G; ++g)
          v[r][g] = sg < nseg ? __ldcg(p.ws_part + (size_t(u) * p.nseg_max + sg) * G + g)
                              : make_float2(-INFINITY, 0.f);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mr = fmaxf(fmaxf(v[0][g].x, v[1][g].x), fmaxf(v[2][g].x, v[3][g].x));
        lse_merge(m[g], s[g], mr, 0.f);        // the lane's max so far, sum rescaled
        const float base = m[g] == -INFINITY ? 0.f : m[g];
#pragma unroll
        for (int r = 0; r < 4; ++r) s[g] += v[r][g].y * __expf(v[r][g].x - base);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float M = m[g];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
      float x = (m[g] == -INFINITY) ? 0.f : s[g] * __expf(m[g] - M);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
      m[g] = M;
      s[g] = x;
    }
    if (wide) {
      __shared__ float2 s_wz[kFinWarps][8];
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) s_wz[tid >> 5][g] = make_float2(m[g], s[g]);
      }
      __syncthreads();
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        s[g] = 0.f;
#pragma unroll
        for (int w = 0; w < kFinWarps; ++w) lse_merge(m[g], s[g], s_wz[w][g].x, s_wz[w][g].y);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
      lz[g] = (s[g] > 0.f && m[g] != -INFINITY) ? m[g] + kLn2 * lg2_approx(s[g]) : -INFINITY;
  }

  // ---- averaged shares m_bar of this slice's candidates (Cor. 3) ------------
  if (select || p.page_share) {
    float lz2[G];
#pragma unroll
    for (int g = 0; g < G; ++g) lz2[g] = lz[g] * kLog2e;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i = kFinThreads * e + tid;
      if (i < c_n) {
        if (!select) ld_scores<G>(ws_s + size_t(1 + c_lo + i) * G, sv[e]);
        float mb = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) mb += ex2_approx(fmaf(sv[e][g], kLog2e, -lz2[g]));
        mb *= 1.f / G;
        keys[i] = __float_as_uint(mb);          // >= 0: the bit pattern orders like the value
        if (p.page_share) p.page_share[size_t(u) * p.max_pages + 1 + c_lo + i] = mb;
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

  // ---- this slice's top-K in page order (between equal shares the smaller
  // page), or all of it when it holds no more than K --------------------------
  auto topk = [&](int m, int KK, auto put) {
    if (KK >= m) {
      for (int i = tid; i < m; i += kFinThreads) put(i, i);
    } else if (m <= kFinThreads) {
      block_topk_small(keys, m, KK, ts.scan[5], put);
    } else {
      block_topk(keys, m, KK, ts, put);
    }
  };
  if (nsl == 1) {
    topk(c_n, K, [=](int i, int pos) { out[1 + pos] = 1 + c_lo + i; });
    if (tid == 0) { out[0] = 0; out[k - 1] = n - 1; }
    return;
  }
  if constexpr (CL) {
    uint2* win = s_win;
    topk(c_n, K, [=](int i, int pos) { win[pos] = make_uint2(keys[i], uint32_t(1 + c_lo + i)); });
    cluster_merge(min(K, c_n));
    return;
  }
  uint2* cand = p.ws_cand + (size_t(u) * p.nslices_max + sl) * p.cand_per_slice;
  topk(c_n, K, [=](int i, int pos) { cand[pos] = make_uint2(keys[i], uint32_t(1 + c_lo + i)); });

  // ---- several slices: the last one selects among the slices' winners -------
  __threadfence();
  __syncthreads();
  if (tid == 0) s_is_last = (atomicAdd(p.ws_ticket + u, 1) == nsl - 1);
  __syncthreads();
  if (!s_is_last) return;
  __threadfence();
  // slice s2 holds min(K, its candidates) winners in page order: K for every
  // slice but the last, so entry i of the concatenation (slice order, still
  // page order) is entry i % K of slice i / K.  All of them load at once.
  const int m_all = (nsl - 1) * K + min(K, n_cand - (nsl - 1) * p.slice);
  for (int i = tid; i < m_all; i += kFinThreads) {
    const int s2 = i / K, e2 = i - s2 * K;
    const uint2 e = __ldcg(p.ws_cand + (size_t(u) * p.nslices_max + s2) * p.cand_per_slice + e2);
    keys[i] = e.x;
    pages[i] = int(e.y);
  }
  __syncthreads();
  topk(m_all, K, [=](int i, int pos) { out[1 + pos] = pages[i]; });
  if (tid == 0) { out[0] = 0; out[k - 1] = n - 1; p.ws_ticket[u] = 0; }
}

template <int G>
int launch_finalize(const SelectParams& p, int n_slices, cudaStream_t stream) {
  const size_t fsmem = size_t(p.fin_cap) * 8;
  if (fsmem + sizeof(TopkScratch) + 6144 > kMaxDynSmem) return LOCKS_ERR_UNSUPPORTED;
  // 2 to 8 slices a unit (portable cluster sizes): one cluster per unit
  const bool cl = n_slices >= 2 && n_slices <= 8;
  auto fk = cl ? finalize_kernel<G, true> : finalize_kernel<G, false>;
  if (cudaFuncSetAttribute(fk, cudaFuncAttributeMaxDynamicSharedMemorySize, int(fsmem)) !=
      cudaSuccess)
    return LOCKS_ERR_CUDA;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(n_slices, p.units);
  lc.blockDim = dim3(kFinThreads);
  lc.dynamicSmemBytes = fsmem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = n_slices;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = cl ? 2 : 1;
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
  g.nseg_max = (g.mc + g.per_cta - 1) / g.per_cta + 1;
  g.slice = kMaxSlice;
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
