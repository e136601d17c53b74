// Split-K paged decode attention over a page list: the selected pages
// (locks_sparse_decode) or every page (locks_dense_decode).  Attention is the
// softmax of q^T k / sqrt(d) over the attended tokens, renormalised over them
// ("Locks: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", section 2 and Lemma 1).
//
// CTA (split s, unit u = (sequence b, KV head h)) handles pages
// [s*P, (s+1)*P) of the unit's page list.  Warp 4 is a producer: its lane 0
// loads each page's K and V (four 64-row x 64-column bf16 boxes through two
// 2-D tensor maps, 128-byte swizzle) into a STAGES-deep shared-memory ring,
// completing on a "full" mbarrier; consumer warps 0..3 release a slot on an
// "empty" mbarrier.  Consumer warp w owns tokens [16w, 16w+16) of every page
// and uses the tensor cores:
//   S (16 x 16)  = Q_pad (16 x 128) . K_w^T       the G query heads are rows
//                                                 0..G-1 of a zero-padded Q
//   O (16 x 128) += P (16 x 16) . V_w (16 x 128)  P re-used from the S
//                                                 accumulators as bf16
// (mma.sync m16n8k16, bf16 inputs, fp32 accumulation; K fragments through
// ldmatrix, V through ldmatrix.trans), with a per-head online softmax (running
// max m, running sum l).  Tokens past the page's valid count are masked and
// their V rows zeroed, so no value outside the sequence enters a product.
// At the end the four warp states are merged into the split's (m, l, acc).
// The splits of a unit are then combined by their log-sum-exp in one of two
// ways:
//   * clustered (page lists of equal length, i.e. the selected pages): the C
//     splits of a unit form one thread-block cluster; each keeps its partial
//     in its own shared memory, and after a cluster barrier CTA r reads all C
//     partials through distributed shared memory and writes its share of the
//     bf16 output rows;
//   * ticketed (every page, lists of unequal length): each split writes its
//     partial to the workspace and the last split of the unit (atomic ticket)
//     brings all of them into shared memory by bulk copies and merges them.
#include <algorithm>

#include "locks_common.cuh"
#include "locks_internal.h"
#include "locks_mma.cuh"

namespace locks {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kDecThreads = (kConsumerWarps + 1) * 32;
constexpr int kTokPerWarp = 16;                            // tokens per consumer warp per stage
constexpr int kStageTokens = kConsumerWarps * kTokPerWarp; // 64
constexpr int kBoxBytes = 64 * 128;                        // 64 rows x 64 bf16
constexpr int kSlotBytes = 4 * kBoxBytes;                  // K0 K1 V0 V1 (32 KiB)
constexpr int kMaxPagesPerSplit = 256;
constexpr int kMaxClusterSplits = 16;                      // cluster size limit (non-portable above 8)
constexpr int kMaxMergeCluster = 4;                        // largest cluster the sparse decode uses

// distributed shared memory: the address of the same variable in CTA `rank`
// of the cluster, and loads from it
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}
// every thread of every CTA of the cluster; shared-memory writes before it are
// visible to the cluster's loads after it
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release;\n"
      "barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void store_out_row(const DecodeParams& p, int b, int h, int G, int gg,
                                              int l4, float4 A, float L, float M) {
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* o = p.out + (size_t(b) * (p.n_kv_heads * G) + h * G + gg) * kHeadDim + 4 * l4;
  const __nv_bfloat162 o01 = __floats2bfloat162_rn(A.x * inv, A.y * inv);
  const __nv_bfloat162 o23 = __floats2bfloat162_rn(A.z * inv, A.w * inv);
  uint2 ow;
  ow.x = *reinterpret_cast<const uint32_t*>(&o01);
  ow.y = *reinterpret_cast<const uint32_t*>(&o23);
  *reinterpret_cast<uint2*>(o) = ow;
  if (l4 == 0 && p.out_lse)
    p.out_lse[size_t(b) * (p.n_kv_heads * G) + h * G + gg] =
        L > 0.f ? M * p.scale + logf(L) : -INFINITY;
}

template <int G, int STAGES, bool CLUSTERED, int PB>
__global__ void __launch_bounds__(kDecThreads)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int u = blockIdx.y, sp = blockIdx.x;
  const int b = u / p.n_kv_heads, h = u % p.n_kv_heads;
  constexpr int B = PB;
  constexpr int PPS = kStageTokens / PB;   // pages per ring stage (1 or 4)

  // ---- shared memory ------------------------------------------------------
  unsigned char* ring = smem;                                       // STAGES x 32 KiB
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(STAGES) * kSlotBytes);
  uint64_t* empty = full + STAGES;
  int* slot_nv = reinterpret_cast<int*>(empty + STAGES);            // [STAGES][4] per warp
  float* wstate = reinterpret_cast<float*>(slot_nv + 4 * STAGES);   // [4][2G]
  __shared__ int s_blk[kMaxPagesPerSplit], s_nv[kMaxPagesPerSplit];
  __shared__ int s_is_last;
  __shared__ uint64_t s_merge_bar;   // the last split's bulk copies of the partials

  // set-up that touches no memory a previous kernel may write runs before
  // the dependency wait
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kConsumerWarps);
    }
    mbar_init(&s_merge_bar, 1);
    mbar_fence_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_k) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_v) : "memory");
  }

  // this sequence's block-table row and length are pulled into L2 while the
  // previous kernel finishes (prefetches return no data, so a writer that is
  // still running cannot be raced), for the page lookups after the wait
  {
    const int32_t* row = p.block_table + size_t(b) * p.max_pages;
    const int lines = (p.max_pages + 31) / 32;     // 128-byte lines of the row
    for (int l = tid; l < lines; l += kDecThreads)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(row + 32 * l));
    if (tid == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.seq_lens + b));
  }

  // launched as a programmatic dependent of the previous kernel on the stream:
  // wait for it to finish before reading anything it may have written
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // the sequence length and (for a selected list, whose length is the same for
  // every unit) this thread's first page id are loaded together
  int seq_len = p.seq_lens[b];
  int j_first = -1;
  if (p.selected) {
    const int lo = sp * p.pages_per_split;
    if (tid < min(p.k, lo + p.pages_per_split) - lo)
      j_first = p.selected[size_t(u) * p.k + lo + tid];
  }
  if (seq_len > p.max_pages * B) {
    if (sp == 0 && tid == 0) flag_status(p.status, LOCKS_DEV_BAD_SEQ_LEN);
    seq_len = p.max_pages * B;
  }
  if (seq_len < 0) seq_len = 0;
  const int n = (seq_len + B - 1) / B;
  const int n_list = p.selected ? p.k : n;
  const int nsplits = CLUSTERED ? int(gridDim.x)
                                : max(1, (n_list + p.pages_per_split - 1) / p.pages_per_split);
  // (a clustered launch has exactly the unit's splits: no CTA leaves early, so
  // every thread reaches the cluster barriers)
  if (!CLUSTERED && sp >= nsplits) return;
  const int i_lo = sp * p.pages_per_split;
  const int cnt = max(0, min(n_list, i_lo + p.pages_per_split) - i_lo);
  const int nst = (cnt + PPS - 1) / PPS;   // ring stages of this split
  // page ids of this split: block and valid tokens, checked once
  const int32_t* bt = p.block_table + size_t(b) * p.max_pages;
  for (int t = tid; t < cnt; t += kDecThreads) {
    const int j = p.selected ? (t == tid ? j_first : p.selected[size_t(u) * p.k + i_lo + t])
                             : i_lo + t;
    int nv = 0, blk = -1;
    if (j >= 0 && j < n) {
      blk = bt[j];
      if (blk >= 0 && blk < p.num_blocks) nv = min(B, seq_len - j * B);
      else flag_status(p.status, LOCKS_DEV_BAD_BLOCK_ID);
    } else if (j >= n) {
      flag_status(p.status, LOCKS_DEV_BAD_PAGE_ID);
    }
    s_blk[t] = blk;
    s_nv[t] = nv;
  }
  __syncthreads();

  // per-lane accumulator of O rows g (= lane / 4) and g + 8, dims 8j + 2t, +1
  float oacc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
  const int g = lane >> 2, t4 = lane & 3;
  float m_run = -INFINITY, l_run = 0.f;            // head g (lanes of a quad agree)

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();   // K/V pages are read once per step
      for (int i = 0; i < nst; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES && !mbar_wait_bounded(empty + s, ((i / STAGES) - 1) & 1)) {
          flag_status(p.status, LOCKS_DEV_WAIT_TIMEOUT);
          break;
        }
        // a stage is 64 token rows: one page (B = 64) or four (B = 16); warp w
        // attends rows [16w, 16w + 16), i.e. its valid count is per warp
        unsigned char* slot = ring + size_t(s) * kSlotBytes;
        uint32_t bytes = 0;
#pragma unroll
        for (int e = 0; e < PPS; ++e) {
          const int t = i * PPS + e;
          if (t < cnt && s_nv[t] > 0) bytes += 2u * PB * kHeadDim * 2u;
        }
        if (PPS == 1) {
          const int nv = s_nv[i];
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w)
            slot_nv[s * 4 + w] = min(kTokPerWarp, max(0, nv - w * kTokPerWarp));
        } else {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const int t = i * PPS + w;
            slot_nv[s * 4 + w] = t < cnt ? s_nv[t] : 0;
          }
        }
        if (bytes) {
          mbar_arrive_expect_tx(full + s, bytes);
#pragma unroll
          for (int e = 0; e < PPS; ++e) {
            const int t = i * PPS + e;
            if (t < cnt && s_nv[t] > 0) {
              const int row = (s_blk[t] * p.n_kv_heads + h) * B;
              unsigned char* dst = slot + e * PB * 128;   // rows [PB e, PB e + PB) of each box
              tma_load_2d(dst, &tmap_k, 0, row, full + s, pol);
              tma_load_2d(dst + kBoxBytes, &tmap_k, 64, row, full + s, pol);
              tma_load_2d(dst + 2 * kBoxBytes, &tmap_v, 0, row, full + s, pol);
              tma_load_2d(dst + 3 * kBoxBytes, &tmap_v, 64, row, full + s, pol);
            }
          }
        } else {
          mbar_arrive(full + s);
        }
      }
    }
  } else {
    // ---------------- consumers ----------------
    // Q fragments (rows = heads, zero beyond G): k-step ks covers dims [16ks, 16ks+16)
    uint32_t qa0[8], qa2[8];
    {
      const __nv_bfloat16* qg = p.q + (size_t(b) * (p.n_kv_heads * G) + h * G + g) * kHeadDim;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa0[ks] = g < G ? *reinterpret_cast<const uint32_t*>(qg + 16 * ks + 2 * t4) : 0u;
        qa2[ks] = g < G ? *reinterpret_cast<const uint32_t*>(qg + 16 * ks + 8 + 2 * t4) : 0u;
      }
    }
    const int n0 = warp * kTokPerWarp;
    int done = nst;
    bool aborted = false;
    for (int i = 0; i < nst; ++i) {
      const int s = i % STAGES;
      if (!__all_sync(kFull, mbar_wait_bounded(full + s, (i / STAGES) & 1))) {
        if (lane == 0) flag_status(p.status, LOCKS_DEV_WAIT_TIMEOUT);
        aborted = true;
        done = i;
        break;
      }
      const int nv = slot_nv[s * 4 + warp];   // valid rows among this warp's 16
      if (nv > 0) {
        const uint32_t kbox = smem_u32(ring + size_t(s) * kSlotBytes);
        const uint32_t vbox = kbox + 2 * kBoxBytes;
        // ---- S = Q K^T over this warp's 16 tokens (two 8-token tiles) ----
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int mi = lane >> 3, r = lane & 7;
          const int tok = n0 + ((mi >> 1) << 3) + r;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            uint32_t kb[4];
            ldsm_x4(swz(kbox + (ks >> 2) * kBoxBytes, tok, 2 * (ks & 3) + (mi & 1)), kb);
            mma16816(sacc[0], qa0[ks], 0u, qa2[ks], 0u, kb[0], kb[1]);
            mma16816(sacc[1], qa0[ks], 0u, qa2[ks], 0u, kb[2], kb[3]);
          }
        }
        // ---- online softmax for head g over rows n0 + {2t, 2t+1, 8+2t, 9+2t} ----
        const int tk0 = 2 * t4;
        float sv[4] = {sacc[0][0], sacc[0][1], sacc[1][0], sacc[1][1]};
        const int tks[4] = {tk0, tk0 + 1, tk0 + 8, tk0 + 9};
        float mt = -INFINITY;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sv[e] = tks[e] < nv ? sv[e] : -INFINITY;
          mt = fmaxf(mt, sv[e]);
        }
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
        const float m_new = fmaxf(m_run, mt);          // finite: the warp has a valid token
        const float alpha = ex2_approx((m_run - m_new) * p.scale_log2);   // 0 when m_run = -inf
        float pr[4], rs = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pr[e] = (g < G) ? ex2_approx((sv[e] - m_new) * p.scale_log2) : 0.f;
          rs += pr[e];
        }
        rs += __shfl_xor_sync(kFull, rs, 1);
        rs += __shfl_xor_sync(kFull, rs, 2);
        l_run = l_run * alpha + rs;
        m_run = m_new;
        if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
          for (int j = 0; j < 16; ++j) { oacc[j][0] *= alpha; oacc[j][1] *= alpha; }
        }
        const uint32_t pa0 = pack_bf16(pr[0], pr[1]), pa2 = pack_bf16(pr[2], pr[3]);
        // ---- tokens past the valid count: zero their V rows (never 0 x NaN) ----
        if (nv < kTokPerWarp) {
          for (int r = n0 + nv; r < n0 + kTokPerWarp; ++r) {
            unsigned char* row0 = ring + size_t(s) * kSlotBytes + 2 * kBoxBytes + r * 128;
            if (lane < 8) *reinterpret_cast<uint4*>(row0 + lane * 16) = make_uint4(0, 0, 0, 0);
            else if (lane < 16)
              *reinterpret_cast<uint4*>(row0 + kBoxBytes + (lane - 8) * 16) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        // ---- O += P V over dims 16j .. 16j+15 ----
        {
          const int mi = lane >> 3, r = lane & 7;
          const int tok = n0 + ((mi & 1) << 3) + r;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t vb[4];
            ldsm_x4_t(swz(vbox + (j >> 2) * kBoxBytes, tok, 2 * (j & 3) + (mi >> 1)), vb);
            mma16816(oacc[2 * j], pa0, 0u, pa2, 0u, vb[0], vb[1]);
            mma16816(oacc[2 * j + 1], pa0, 0u, pa2, 0u, vb[2], vb[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
    }
    if (aborted) {
      for (int i = done; i < min(nst, done + STAGES); ++i)
        mbar_wait_bounded(full + (i % STAGES), (i / STAGES) & 1);
    }
  }
  __syncthreads();

  // ---- merge the four warp states into the split's partial ----------------
  float* mbuf = reinterpret_cast<float*>(ring);    // [4][G][128], the ring is idle now
  if (warp < kConsumerWarps) {
    if (g < G) {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        *reinterpret_cast<float2*>(mbuf + (warp * G + g) * kHeadDim + 8 * j + 2 * t4) =
            make_float2(oacc[j][0], oacc[j][1]);
      if (t4 == 0) {
        wstate[warp * 2 * G + g] = m_run;
        wstate[warp * 2 * G + G + g] = l_run;
      }
    }
  }
  __syncthreads();
  const size_t part_stride = kPartStride;   // [m, l, pad, pad, acc[d]]: acc 16-byte aligned
  // the split's partial: in this CTA's shared memory (clustered), past the
  // warp accumulators in the idle ring, or in the workspace (ticketed)
  float* part = CLUSTERED
                    ? reinterpret_cast<float*>(ring + kConsumerWarps * G * kHeadDim * sizeof(float))
                    : p.ws_part + (size_t(u) * p.n_splits_max + sp) * G * part_stride;
  for (int t = tid; t < G * 32; t += kDecThreads) {
    const int gg = t >> 5, l4 = t & 31;
    float M = -INFINITY;
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wstate[w * 2 * G + gg]);
    float L = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = wstate[w * 2 * G + gg];
        if (mw == -INFINITY) continue;
        const float f = exp2f((mw - M) * p.scale_log2);
        L += wstate[w * 2 * G + G + gg] * f;
        const float4 a = *reinterpret_cast<const float4*>(mbuf + (w * G + gg) * kHeadDim + 4 * l4);
        A.x += a.x * f; A.y += a.y * f; A.z += a.z * f; A.w += a.w * f;
      }
    }
    float* pg = part + gg * part_stride;
    if (l4 == 0) { pg[0] = M; pg[1] = L; }
    *reinterpret_cast<float4*>(pg + 4 + 4 * l4) = A;
  }

  if constexpr (CLUSTERED) {
    // ---- merge the unit's splits through distributed shared memory ----------
    // CTA sp writes output entries [sp * per, (sp + 1) * per) of the unit's
    // G x 32 (head, 4-dim chunk) entries
    __syncthreads();
    cluster_sync_all();
    const int C = nsplits;
    const int per = (G * 32 + C - 1) / C;
    const int t_end = min(G * 32, (sp + 1) * per);
    for (int t = sp * per + tid; t < t_end; t += kDecThreads) {
      const int gg = t >> 5, l4 = t & 31;
      const uint32_t a_ml = smem_u32(part + gg * part_stride);
      const uint32_t a_acc = a_ml + (4 + 4 * l4) * sizeof(float);
      float2 ml[kMaxClusterSplits];
      float4 ac[kMaxClusterSplits];
#pragma unroll
      for (int r = 0; r < kMaxClusterSplits; ++r) {
        if (r < C) {
          ml[r] = ld_dsmem_f2(dsmem_addr(a_ml, r));
          ac[r] = ld_dsmem_f4(dsmem_addr(a_acc, r));
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxClusterSplits; ++r)
        if (r < C) M = fmaxf(M, ml[r].x);
      float L = 0.f;
      float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
#pragma unroll
        for (int r = 0; r < kMaxClusterSplits; ++r) {
          if (r < C && ml[r].x != -INFINITY) {
            const float f = exp2f((ml[r].x - M) * p.scale_log2);
            L += ml[r].y * f;
            A.x += ac[r].x * f; A.y += ac[r].y * f; A.z += ac[r].z * f; A.w += ac[r].w * f;
          }
        }
      }
      store_out_row(p, b, h, G, gg, l4, A, L, M);
    }
    // no CTA leaves while another may still read its shared memory
    cluster_sync_all();
    return;
  }

  __threadfence();
  __syncthreads();
  if (tid == 0) s_is_last = (atomicAdd(p.ws_ticket + u, 1) == nsplits - 1);
  __syncthreads();
  if (!s_is_last) return;
  __threadfence();

  // ---- last split of the unit: merge every split -----------------------------
  // The unit's partials (nsplits x G x kPartStride floats) are contiguous in
  // the workspace: they come into the idle ring by one bulk copy per chunk of
  // as many splits as it holds, so every load is in flight at once; each
  // thread merges its output entries' (m, l, acc) from shared memory, per
  // chunk by its maximum first, then into a running state.
  constexpr int kItems = (G * 32 + kDecThreads - 1) / kDecThreads;
  const uint32_t split_bytes = uint32_t(G * part_stride * sizeof(float));
  const int cap = int((size_t(STAGES) * kSlotBytes) / split_bytes);
  const float* src = p.ws_part + size_t(u) * p.n_splits_max * G * part_stride;
  const float* buf = reinterpret_cast<const float*>(ring);
  float rM[kItems], rL[kItems];
  float4 rA[kItems];
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    rM[it] = -INFINITY;
    rL[it] = 0.f;
    rA[it] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  bool merge_ok = true;
  int ph = 0;
  for (int c0 = 0; c0 < nsplits && merge_ok; c0 += cap, ++ph) {
    const int cn = min(cap, nsplits - c0);
    if (tid == 0) {
      // the other splits' partials were written through the generic proxy (and
      // made visible by their fences and the ticket); order them, and this
      // CTA's earlier use of the ring, before the copy engine's accesses
      asm volatile("fence.proxy.async.global;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&s_merge_bar, uint32_t(cn) * split_bytes);
      bulk_g2s(ring, src + size_t(c0) * G * part_stride, uint32_t(cn) * split_bytes, &s_merge_bar);
    }
    // every thread waits; the block agrees on the outcome before any leaves
    const bool landed = mbar_wait_bounded(&s_merge_bar, ph & 1);
    if (__syncthreads_or(!landed)) {
      if (tid == 0) flag_status(p.status, LOCKS_DEV_WAIT_TIMEOUT);
      merge_ok = false;
      break;
    }
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int t = tid + it * kDecThreads;
      if (t >= G * 32) break;
      const int gg = t >> 5, l4 = t & 31;
      float Mc = -INFINITY;
      for (int s2 = 0; s2 < cn; ++s2) Mc = fmaxf(Mc, buf[(s2 * G + gg) * part_stride]);
      if (Mc == -INFINITY) continue;
      float Lc = 0.f;
      float4 Ac = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int s2 = 0; s2 < cn; ++s2) {
        const float* pg = buf + (s2 * G + gg) * part_stride;
        const float2 ml = *reinterpret_cast<const float2*>(pg);
        const float4 a2 = *reinterpret_cast<const float4*>(pg + 4 + 4 * l4);
        const float f = ml.x == -INFINITY ? 0.f : exp2f((ml.x - Mc) * p.scale_log2);
        Lc += ml.y * f;
        Ac.x += a2.x * f; Ac.y += a2.y * f; Ac.z += a2.z * f; Ac.w += a2.w * f;
      }
      const float Mn = fmaxf(rM[it], Mc);
      const float fo = rM[it] == -INFINITY ? 0.f : exp2f((rM[it] - Mn) * p.scale_log2);
      const float fc = exp2f((Mc - Mn) * p.scale_log2);
      rL[it] = rL[it] * fo + Lc * fc;
      rA[it].x = rA[it].x * fo + Ac.x * fc;
      rA[it].y = rA[it].y * fo + Ac.y * fc;
      rA[it].z = rA[it].z * fo + Ac.z * fc;
      rA[it].w = rA[it].w * fo + Ac.w * fc;
      rM[it] = Mn;
    }
    __syncthreads();                               // the next chunk overwrites the ring
  }
  if (!merge_ok) {
    // let the copy in flight land before the CTA can exit
    mbar_wait_bounded(&s_merge_bar, ph & 1);
  } else {
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int t = tid + it * kDecThreads;
      if (t < G * 32) store_out_row(p, b, h, G, t >> 5, t & 31, rA[it], rL[it], rM[it]);
    }
  }
  if (tid == 0) p.ws_ticket[u] = 0;
}

template <int G>
constexpr size_t decode_smem_bytes(int stages) {
  return size_t(stages) * kSlotBytes + 2 * stages * sizeof(uint64_t) + 4 * stages * sizeof(int) +
         kConsumerWarps * 2 * G * sizeof(float);
}

// How many clusters of C decode CTAs this device can hold at once (0: none;
// queried once per group size, page size and cluster size).
template <int G, int PB>
int cluster_capacity(int C) {
  static int known[kMaxClusterSplits + 1] = {};   // 0 unknown, else capacity + 1
  if (C < 1 || C > kMaxClusterSplits) return 0;
  const int k = __atomic_load_n(&known[C], __ATOMIC_ACQUIRE);
  if (k != 0) return k - 1;
  constexpr int STAGES = 3;
  auto kern = decode_kernel<G, STAGES, true, PB>;
  const size_t smem = decode_smem_bytes<G>(STAGES);
  bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) ==
                cudaSuccess &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                cudaSuccess;
  int n_clusters = 0;
  if (ok) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(C, 1);
    lc.blockDim = dim3(kDecThreads);
    lc.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    ok = cudaOccupancyMaxActiveClusters(&n_clusters, kern, &lc) == cudaSuccess;
  }
  if (!ok) {
    cudaGetLastError();            // a refused query leaves no error behind
    n_clusters = 0;
  }
  __atomic_store_n(&known[C], n_clusters + 1, __ATOMIC_RELEASE);
  return n_clusters;
}

template <int G, int PB>
int launch_g(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int gx, int gy,
             bool clustered, cudaStream_t stream) {
  constexpr int STAGES = 3;
  const size_t smem = decode_smem_bytes<G>(STAGES);
  auto kern = clustered ? decode_kernel<G, STAGES, true, PB> : decode_kernel<G, STAGES, false, PB>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return LOCKS_ERR_CUDA;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(gx, gy);
  lc.blockDim = dim3(kDecThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = gx;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = clustered ? 2 : 1;
  return cudaLaunchKernelEx(&lc, kern, p, tk, tv) == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
}

template <int G, int PB>
int launch_list(DecodeParams p, const CUtensorMap& tk, const CUtensorMap& tv, int gx, int gy,
                cudaStream_t stream) {
  if (p.selected && p.k > 0) {
    // equal-length lists: one cluster of at most kMaxClusterSplits splits per
    // unit, each split a whole number of ring stages
    constexpr int PPS = kStageTokens / PB;
    // Few units (at most 16, as at a million tokens with one sequence): the
    // decode is a latency chain, and clusters of up to 8 splits of several
    // pages, merged on chip, end it sooner than a ticketed merge of many
    // one-page splits (1M: 1 us per step).  More units: only small clusters
    // (at most kMaxMergeCluster CTAs): in a decode step, which starts while
    // the selection's kernels still hold SMs, larger clusters were measured to
    // start late (32 units in clusters of 8: 5 us slower per step than the
    // ticketed merge of the same 8 splits).
    const bool few_units = gy <= 16;
    const int cap = few_units ? 8 : kMaxMergeCluster;
    const int most = few_units ? 8 : kMaxClusterSplits;
    int pps = std::max(p.pages_per_split, (p.k + most - 1) / most);
    pps = (pps + PPS - 1) / PPS * PPS;
    const int C = (p.k + pps - 1) / pps;
    if (C <= cap && cluster_capacity<G, PB>(C) > 0) {
      p.pages_per_split = pps;
      return launch_g<G, PB>(p, tk, tv, C, gy, true, stream);
    }
  }
  return launch_g<G, PB>(p, tk, tv, gx, gy, false, stream);
}

template <int PB>
int launch_pb(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int G, int gx,
              int gy, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_list<1, PB>(p, tk, tv, gx, gy, stream);
    case 2: return launch_list<2, PB>(p, tk, tv, gx, gy, stream);
    case 4: return launch_list<4, PB>(p, tk, tv, gx, gy, stream);
    case 8: return launch_list<8, PB>(p, tk, tv, gx, gy, stream);
    default: return LOCKS_ERR_UNSUPPORTED;
  }
}

}  // namespace

int decode_pages_per_split(long units, int n_pages, int page_size) {
  // in ring stages of 64 tokens (one page of 64, four of 16): a whole number
  // of splits per unit such that all splits fit one wave of two CTAs per SM on
  // 152 SMs (two waves for long lists); at most kMaxPagesPerSplit pages per CTA
  const long pps_stage = page_size > 0 && page_size < kStageTokens ? kStageTokens / page_size : 1;
  const long np = n_pages > 0 ? (n_pages + pps_stage - 1) / pps_stage : 1;
  const long waves = units * np > 16384 ? 2 : 1;
  long splits = (waves * 2 * 152) / (units > 0 ? units : 1);
  if (splits < 1) splits = 1;
  long st = (np + splits - 1) / splits;
  if (st * pps_stage > kMaxPagesPerSplit) st = kMaxPagesPerSplit / pps_stage;
  return int(st * pps_stage);
}

int launch_decode(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int G,
                  int gx, int gy, cudaStream_t stream) {
  if (p.page_size == 64) return launch_pb<64>(p, tk, tv, G, gx, gy, stream);
  if (p.page_size == 16) return launch_pb<16>(p, tk, tv, G, gx, gy, stream);
  return LOCKS_ERR_UNSUPPORTED;
}

}  // namespace locks
