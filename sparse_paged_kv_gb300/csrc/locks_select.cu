// locks_select: page scoring (Eq. (1)), per-head page-mass shares, the GQA
// share-average and the forced-page top-(k-2) selection of
// "Locks: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", section 4 ("Score") and Cor. 3.
//
// One grid covers every (sequence b, KV head h) "unit".  CTA (c, u) scores
// the c-th chunk of unit u's candidate pages.  Each warp owns a ring of
// STAGES shared-memory slots; lane 0 streams the page summary records of the
// warp's pages into them with 1-D bulk copies, and the whole warp scores one
// page per step:
//
//   lane l holds dims [4l, 4l+4) of the G group queries, dots them with the
//   centroid and basis rows (a_g = q_g.mu, p_gk = q_g.v_k), the G*R partial
//   dot products are reduced across the warp with a transposed reduction,
//   broadcast through shared memory, and lane l then forms the reconstructed
//   logits of tokens l and l+32 for every head and reduces them by
//   log-sum-exp.
//
// The CTA writes s_hat per (page, head) and its chunk's per-head (max, sum)
// log-sum-exp partial.  The last CTA of a unit to finish (an atomic ticket,
// no waiting) merges the partials into log Z_g, forms the averaged shares
// m_bar_j of every candidate, finds the (k-2)-th largest by a 4-pass 8-bit
// radix select over the share bit patterns, and writes the ascending page list.
#include "locks_common.cuh"
#include "locks_internal.h"

namespace locks {

namespace {

constexpr int kSelWarps = 8;
constexpr int kSelThreads = kSelWarps * 32;

// floats of per-warp broadcast buffer: G*R projections + G centroid terms,
// padded to 16 bytes
template <int G, int RP>
__host__ __device__ constexpr int pbuf_stride() { return (G * RP + G + 3) / 4 * 4; }

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Block-wide exclusive scan of one int per thread; returns the exclusive
// prefix and writes the block total to *total.  `scratch` holds >= 32 ints.
__device__ int block_excl_scan(int x, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int incl = warp_incl_scan(x, lane);
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < kSelWarps ? scratch[lane] : 0;
    const int vi = warp_incl_scan(v, lane);
    if (lane < kSelWarps) scratch[lane] = vi - v;
    if (lane == kSelWarps - 1) scratch[kSelWarps] = vi;
  }
  __syncthreads();
  const int res = scratch[warp] + incl - x;
  *total = scratch[kSelWarps];
  __syncthreads();
  return res;
}

// Scores one page summary `rec` for the G queries held in qv (dims [4l,4l+4)).
// Returns the G scores s_hat (identical in every lane).
template <int G, int RP, typename T>
__device__ __forceinline__ void score_page(const T* __restrict__ rec, const float4 (&qv)[G],
                                           float* pbuf, int lane, float scale, float scale_log2,
                                           float (&shat)[G]) {
  constexpr int NP = G * RP;                   // basis projections p_{g,k}
  constexpr int SP = NP < 32 ? NP : 32;
  constexpr int VP = NP / SP;                  // values a lane holds after the reduction
  constexpr int SA = G < 32 ? G : 32;

  float pv[NP];
  float av[G];
  {
    const float4 w = ld4(rec + 4 * lane);      // centroid row
#pragma unroll
    for (int g = 0; g < G; ++g)
      av[g] = qv[g].x * w.x + qv[g].y * w.y + qv[g].z * w.z + qv[g].w * w.w;
  }
#pragma unroll
  for (int k = 0; k < RP; ++k) {
    const float4 w = ld4(rec + (1 + k) * kHeadDim + 4 * lane);
#pragma unroll
    for (int g = 0; g < G; ++g)
      pv[g * RP + k] = qv[g].x * w.x + qv[g].y * w.y + qv[g].z * w.z + qv[g].w * w.w;
  }
  TransposeReduce<NP, 16>::run(pv, lane);
  TransposeReduce<G, 16>::run(av, lane);
  // lane l now holds p values [(l / (32/SP)) * VP, +VP) and a value l / (32/SA)
  if ((lane & (32 / SP - 1)) == 0) {
#pragma unroll
    for (int e = 0; e < VP; ++e) pbuf[(lane / (32 / SP)) * VP + e] = pv[e];
  }
  if ((lane & (32 / SA - 1)) == 0) pbuf[NP + lane / (32 / SA)] = av[0];
  __syncwarp();

  // reconstructed logits (before the 1/sqrt(d) scale) of tokens lane, lane+32
  const T* C = rec + rec_w_elems(RP);
  float x[G][2];
#pragma unroll
  for (int g = 0; g < G; ++g) x[g][0] = x[g][1] = 0.f;
#pragma unroll
  for (int cc = 0; cc < RP / 4; ++cc) {
    const float4 c0 = ld4(C + (cc * kPageSize + lane) * 4);
    const float4 c1 = ld4(C + (cc * kPageSize + lane + 32) * 4);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float4 p = *reinterpret_cast<const float4*>(pbuf + g * RP + cc * 4);
      x[g][0] += p.x * c0.x + p.y * c0.y + p.z * c0.z + p.w * c0.w;
      x[g][1] += p.x * c1.x + p.y * c1.y + p.z * c1.z + p.w * c1.w;
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float m = group_max<32>(fmaxf(x[g][0], x[g][1]));
    const float e = exp2f((x[g][0] - m) * scale_log2) + exp2f((x[g][1] - m) * scale_log2);
    const float s = group_sum<32>(e);
    shat[g] = scale * (pbuf[NP + g] + m) + logf(s);
  }
  __syncwarp();   // pbuf is rewritten by the next page
}

template <int G, int RP, typename T, int STAGES>
__global__ void __launch_bounds__(kSelThreads)
    select_kernel(const SelectParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int u = blockIdx.y, chunk = blockIdx.x;
  const int b = u / p.n_kv_heads, h = u % p.n_kv_heads;
  const int B = kPageSize;

  // ---- the unit's candidate pages ---------------------------------------
  int seq_len = p.seq_lens[b];
  if (seq_len > p.max_pages * B) {
    if (chunk == 0 && tid == 0) flag_status(p.status, LOCKS_DEV_BAD_SEQ_LEN);
    seq_len = p.max_pages * B;
  }
  if (seq_len < 0) seq_len = 0;
  const int n = (seq_len + B - 1) / B;
  const int n_complete = seq_len / B;
  const int cand_hi = min(n - 1, n_complete);          // candidates are pages 1 .. cand_hi-1
  const int n_cand = max(0, cand_hi - 1);
  const int nchunks = max(1, (n_cand + p.chunk_pages - 1) / p.chunk_pages);
  if (chunk >= nchunks) return;
  const int c_lo = chunk * p.chunk_pages;
  const int c_hi = min(n_cand, c_lo + p.chunk_pages);

  // ---- shared memory ------------------------------------------------------
  const size_t rec_bytes = p.rec_bytes;
  unsigned char* ring = smem;
  const size_t ring_bytes = size_t(kSelWarps) * STAGES * rec_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_bytes);
  float* pbuf_all = reinterpret_cast<float*>(bars + kSelWarps * STAGES);
  float* pbuf = pbuf_all + warp * pbuf_stride<G, RP>();
  float2* wpart = reinterpret_cast<float2*>(pbuf_all + kSelWarps * pbuf_stride<G, RP>());
  __shared__ float s_logz[16];
  __shared__ int s_is_last;

  uint64_t* mybar = bars + warp * STAGES;
  unsigned char* myring = ring + size_t(warp) * STAGES * rec_bytes;
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(mybar + s, 1);
    mbar_fence_init();
  }
  __syncwarp();

  // group queries, dims [4*lane, 4*lane+4)
  float4 qv[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint2 w = *reinterpret_cast<const uint2*>(
        p.q + (size_t(b) * (p.n_kv_heads * G) + h * G + g) * kHeadDim + 4 * lane);
    qv[g] = bf16x4_to_f4(w);
  }

  const int my_count = (c_hi - c_lo - warp + kSelWarps - 1) / kSelWarps;   // may be <= 0
  const int32_t* bt = p.block_table + size_t(b) * p.max_pages;
  const unsigned char* sum_base = static_cast<const unsigned char*>(p.summaries);

  auto page_of = [&](int i) { return 1 + c_lo + warp + i * kSelWarps; };
  auto issue = [&](int i) {
    const int s = i % STAGES;
    const int j = page_of(i);
    const int blk = bt[j];
    if (blk >= 0 && blk < p.num_blocks) {
      mbar_arrive_expect_tx(mybar + s, uint32_t(rec_bytes));
      bulk_g2s(myring + size_t(s) * rec_bytes,
               sum_base + (size_t(blk) * p.n_kv_heads + h) * rec_bytes, uint32_t(rec_bytes),
               mybar + s);
    } else {
      flag_status(p.status, LOCKS_DEV_BAD_BLOCK_ID);
      mbar_arrive(mybar + s);
    }
  };
  if (lane == 0)
    for (int i = 0; i < min(STAGES, my_count); ++i) issue(i);

  // running log-sum-exp of s_hat over this warp's pages; lane g < G tracks head g
  float zm = -INFINITY, zs = 0.f;
  float* ws_s = p.ws_scores + size_t(u) * p.max_pages * G;
  bool aborted = false;
  int done = 0;
  for (int i = 0; i < my_count; ++i) {
    const int s = i % STAGES;
    const bool ok = __all_sync(kFull, mbar_wait_bounded(mybar + s, (i / STAGES) & 1));
    if (!ok) {
      if (lane == 0) flag_status(p.status, LOCKS_DEV_WAIT_TIMEOUT);
      aborted = true;
      done = i;
      break;
    }
    const int j = page_of(i);
    const int blk = bt[j];
    float shat[G];
    if (blk >= 0 && blk < p.num_blocks) {
      score_page<G, RP, T>(reinterpret_cast<const T*>(myring + size_t(s) * rec_bytes), qv, pbuf,
                           lane, p.scale, p.scale_log2, shat);
    } else {
#pragma unroll
      for (int g = 0; g < G; ++g) shat[g] = -INFINITY;
    }
    // lane g writes head g's score; every lane keeps its head's running LSE
    float mine = shat[0];
#pragma unroll
    for (int g = 1; g < G; ++g)
      if (lane == g) mine = shat[g];
    if (lane < G) {
      ws_s[size_t(j) * G + lane] = mine;
      if (p.page_lse)
        p.page_lse[(size_t(b) * (p.n_kv_heads * G) + h * G + lane) * p.max_pages + j] = mine;
      lse_merge(zm, zs, mine, 1.f);
    }
    __syncwarp();
    if (lane == 0 && i + STAGES < my_count) issue(i + STAGES);
  }
  if (aborted) {
    // let the copies still in flight land before the CTA can exit
    for (int i = done; i < min(my_count, done + STAGES); ++i)
      mbar_wait_bounded(mybar + (i % STAGES), (i / STAGES) & 1);
  }

  // ---- chunk partial of log Z -------------------------------------------
  if (lane < G) wpart[warp * G + lane] = make_float2(zm, zs);
  __syncthreads();
  if (tid < G) {
    float m = -INFINITY, sm = 0.f;
    for (int w = 0; w < kSelWarps; ++w) {
      const float2 v = wpart[w * G + tid];
      lse_merge(m, sm, v.x, v.y);
    }
    p.ws_part[(size_t(u) * p.n_chunks_max + chunk) * G + tid] = make_float2(m, sm);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int ticket = atomicAdd(p.ws_ticket + u, 1);
    s_is_last = (ticket == nchunks - 1);
  }
  __syncthreads();
  if (!s_is_last) return;
  __threadfence();

  // ======== last CTA of the unit: normalise, share-average, top-(k-2) =========
  if (tid < G) {
    float m = -INFINITY, sm = 0.f;
    for (int c = 0; c < nchunks; ++c) {
      const float2 v = __ldcg(p.ws_part + (size_t(u) * p.n_chunks_max + c) * G + tid);
      lse_merge(m, sm, v.x, v.y);
    }
    s_logz[tid] = (sm > 0.f) ? m + logf(sm) : -INFINITY;
  }
  __syncthreads();

  const int k = p.k;
  int32_t* out = p.selected + size_t(u) * k;
  if (n <= k) {
    for (int t = tid; t < k; t += kSelThreads) out[t] = t < n ? t : -1;
    if (tid == 0) p.ws_ticket[u] = 0;
    // shares are still reported for the candidates
    for (int idx = tid; idx < n_cand; idx += kSelThreads) {
      const int j = 1 + idx;
      float mb = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) mb += expf(__ldcg(ws_s + size_t(j) * G + g) - s_logz[g]);
      if (p.page_share) p.page_share[size_t(u) * p.max_pages + j] = mb / G;
    }
    return;
  }

  // the barriers' memory may be reused for the keys below
  if (lane == 0)
    for (int s = 0; s < STAGES; ++s)
      asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(mybar + s)) : "memory");
  __syncthreads();
  const int K = k - 2;
  if (K == 0) {
    if (tid == 0) { out[0] = 0; out[1] = n - 1; p.ws_ticket[u] = 0; }
    return;
  }

  // averaged shares as sortable keys (non-negative floats order as their bits)
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  for (int idx = tid; idx < n_cand; idx += kSelThreads) {
    const int j = 1 + idx;
    float mb = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) mb += expf(__ldcg(ws_s + size_t(j) * G + g) - s_logz[g]);
    mb *= 1.f / G;
    keys[idx] = __float_as_uint(mb);
    if (p.page_share) p.page_share[size_t(u) * p.max_pages + j] = mb;
  }
  __syncthreads();

  // radix select of the K-th largest key
  __shared__ unsigned int hist[256];
  __shared__ unsigned int s_digit, s_above;
  __shared__ int scan_scratch[kSelWarps + 1];
  uint32_t prefix = 0, mask = 0;
  int kleft = K;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int t = tid; t < 256; t += kSelThreads) hist[t] = 0;
    __syncthreads();
    for (int idx = tid; idx < n_cand; idx += kSelThreads) {
      const uint32_t key = keys[idx];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins [8*(31-l), 8*(31-l)+8): lane 0 the highest
      unsigned int cnt[8], tot = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cnt[e] = hist[8 * (31 - lane) + 7 - e];   // descending bin order
        tot += cnt[e];
      }
      const int incl = warp_incl_scan(int(tot), lane);
      const int excl = incl - int(tot);
      const unsigned int hit = __ballot_sync(kFull, incl >= kleft);
      const int first = __ffs(hit) - 1;
      if (lane == first) {
        int acc = excl;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (acc + int(cnt[e]) >= kleft) {
            s_digit = 8 * (31 - lane) + 7 - e;
            s_above = acc;
            break;
          }
          acc += cnt[e];
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    kleft -= int(s_above);
    __syncthreads();
  }
  const uint32_t thr = prefix;   // the K-th largest key
  const int need = kleft;        // keys equal to thr to take (the lowest page ids)

  // collect: contiguous index ranges per thread keep the output ordered
  const int per = (n_cand + kSelThreads - 1) / kSelThreads;
  const int lo = min(n_cand, tid * per), hi = min(n_cand, lo + per);
  int n_eq = 0;
  for (int idx = lo; idx < hi; ++idx) n_eq += keys[idx] == thr;
  int tot_eq;
  const int eq_before = block_excl_scan(n_eq, scan_scratch, &tot_eq);
  int n_sel = 0;
  {
    int e = eq_before;
    for (int idx = lo; idx < hi; ++idx) {
      const uint32_t key = keys[idx];
      if (key > thr) ++n_sel;
      else if (key == thr) { if (e < need) ++n_sel; ++e; }
    }
  }
  int tot_sel;
  int pos = block_excl_scan(n_sel, scan_scratch, &tot_sel);
  {
    int e = eq_before;
    for (int idx = lo; idx < hi; ++idx) {
      const uint32_t key = keys[idx];
      bool take = false;
      if (key > thr) take = true;
      else if (key == thr) { take = e < need; ++e; }
      if (take) out[1 + pos++] = 1 + idx;
    }
  }
  if (tid == 0) {
    out[0] = 0;
    out[k - 1] = n - 1;
    p.ws_ticket[u] = 0;   // ready for the next call
  }
}

template <int G, int RP, typename T>
int launch_select_t(const SelectParams& p, int grid_x, int grid_y, cudaStream_t stream) {
  constexpr int STAGES = 2;
  size_t ring = size_t(kSelWarps) * STAGES * p.rec_bytes;
  size_t smem = ring + kSelWarps * STAGES * sizeof(uint64_t) +
                kSelWarps * pbuf_stride<G, RP>() * sizeof(float) + kSelWarps * G * sizeof(float2);
  const size_t keys = size_t(p.max_pages) * sizeof(uint32_t);
  if (keys > smem) smem = keys;
  if (smem > kMaxDynSmem) return LOCKS_ERR_UNSUPPORTED;
  auto kern = select_kernel<G, RP, T, STAGES>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return LOCKS_ERR_CUDA;
  kern<<<dim3(grid_x, grid_y), kSelThreads, smem, stream>>>(p);
  return cudaPeekAtLastError() == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
}

template <typename T>
int dispatch_g(const SelectParams& p, int G, int RP, int gx, int gy, cudaStream_t s) {
#define LOCKS_SEL_CASE(GG, RR)                                \
  if (G == GG && RP == RR) return launch_select_t<GG, RR, T>(p, gx, gy, s);
  LOCKS_SEL_CASE(1, 4) LOCKS_SEL_CASE(1, 8) LOCKS_SEL_CASE(1, 16)
  LOCKS_SEL_CASE(2, 4) LOCKS_SEL_CASE(2, 8) LOCKS_SEL_CASE(2, 16)
  LOCKS_SEL_CASE(4, 4) LOCKS_SEL_CASE(4, 8) LOCKS_SEL_CASE(4, 16)
  LOCKS_SEL_CASE(8, 4) LOCKS_SEL_CASE(8, 8) LOCKS_SEL_CASE(8, 16)
#undef LOCKS_SEL_CASE
  return LOCKS_ERR_UNSUPPORTED;
}

}  // namespace

int select_chunk_pages(int max_pages) {
  // candidates per CTA: enough chunks for several waves, at least 2 pages/warp
  (void)max_pages;
  return 8 * kSelWarps;
}

int launch_select(const SelectParams& p, int G, int RP, int dtype, int grid_x, int grid_y,
                  cudaStream_t stream) {
  if (dtype == LOCKS_SUMMARY_F32) return dispatch_g<float>(p, G, RP, grid_x, grid_y, stream);
  return dispatch_g<__nv_bfloat16>(p, G, RP, grid_x, grid_y, stream);
}

}  // namespace locks
