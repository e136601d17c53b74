// Split-K paged decode attention over a page list: the selected pages
// (locks_sparse_decode) or every page (locks_dense_decode).  Attention is the
// softmax of q^T k / sqrt(d) over the attended tokens, renormalised over them
// ("Locks: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", section 2 and Lemma 1).
//
// CTA (split s, unit u = (sequence b, KV head h)) handles pages
// [s*P, (s+1)*P) of the unit's page list.  Warp 4 is a producer: its lane 0
// bulk-copies the valid token rows of each page's K and V (contiguous
// [B][d] bf16 rows in the pool) into a STAGES-deep shared-memory ring,
// completing on a "full" mbarrier; consumer warps 0..3 release a slot on an
// "empty" mbarrier.  Consumer warp w owns tokens [16w, 16w+16) of every page
// and keeps, for each of the G query heads of the group, a running max m,
// running sum l and an unnormalised output accumulator (dims [4l, 4l+4) in
// lane l).  Scores: 8 lanes per token (16 dims each), 4 tokens per step,
// reduced with a transposed 8-lane reduction.  At the end the four warp states
// are merged, the split writes (m, l, acc) to the workspace, and the last split
// of the unit (atomic ticket) merges all splits by their log-sum-exp and writes
// the bf16 output and the natural-log lse.
#include "locks_common.cuh"
#include "locks_internal.h"

namespace locks {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kDecThreads = (kConsumerWarps + 1) * 32;
constexpr int kTokPerWarp = kPageSize / kConsumerWarps;    // 16
constexpr int kRowBytes = kHeadDim * 2;                    // 256
constexpr int kPageBytes = kPageSize * kRowBytes;          // 16 KiB
constexpr int kSlotBytes = 2 * kPageBytes;                 // K then V

constexpr int kMaxPagesPerSplit = 64;

// float max through the integer atomics (ordering of IEEE bit patterns)
__device__ __forceinline__ void atomicMax_float(float* addr, float v) {
  if (v >= 0.f) atomicMax(reinterpret_cast<int*>(addr), __float_as_int(v));
  else atomicMin(reinterpret_cast<unsigned int*>(addr), __float_as_uint(v));
}

template <int G>
__host__ __device__ constexpr int warp_buf_floats() {
  return ((2 * G * kTokPerWarp + 3 * G) + 3) / 4 * 4;
}

template <int G, int STAGES>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int u = blockIdx.y, sp = blockIdx.x;
  const int b = u / p.n_kv_heads, h = u % p.n_kv_heads;
  constexpr int B = kPageSize;

  // launched as a programmatic dependent of the previous kernel on the stream:
  // wait for it to finish before reading anything it may have written
  asm volatile("griddepcontrol.wait;" ::: "memory");

  int seq_len = p.seq_lens[b];
  if (seq_len > p.max_pages * B) {
    if (sp == 0 && tid == 0) flag_status(p.status, LOCKS_DEV_BAD_SEQ_LEN);
    seq_len = p.max_pages * B;
  }
  if (seq_len < 0) seq_len = 0;
  const int n = (seq_len + B - 1) / B;
  const int n_list = p.selected ? p.k : n;
  const int nsplits = max(1, (n_list + p.pages_per_split - 1) / p.pages_per_split);
  if (sp >= nsplits) return;
  const int i_lo = sp * p.pages_per_split;
  const int cnt = max(0, min(n_list, i_lo + p.pages_per_split) - i_lo);

  // ---- shared memory ------------------------------------------------------
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(STAGES) * kSlotBytes);
  uint64_t* empty = full + STAGES;
  int* slot_nv = reinterpret_cast<int*>(empty + STAGES);
  float* wbuf_all = reinterpret_cast<float*>(slot_nv + ((STAGES + 3) / 4) * 4);
  __shared__ int s_is_last;

  __shared__ int s_blk[kMaxPagesPerSplit], s_nv[kMaxPagesPerSplit];
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kConsumerWarps);
    }
    mbar_fence_init();
  }
  // page ids of this split: block and valid tokens, checked once
  const int32_t* bt = p.block_table + size_t(b) * p.max_pages;
  for (int t = tid; t < cnt; t += kDecThreads) {
    const int j = p.selected ? p.selected[size_t(u) * p.k + i_lo + t] : i_lo + t;
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

  float acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) acc[g][0] = acc[g][1] = acc[g][2] = acc[g][3] = 0.f;
  float* wb = wbuf_all + warp * warp_buf_floats<G>();
  float* s_buf = wb;                              // [G][16] raw scores
  float* p_buf = wb + G * kTokPerWarp;            // [16][G] probabilities
  float* run_m = p_buf + G * kTokPerWarp;         // [G]
  float* run_l = run_m + G;                       // [G]
  float* alpha_buf = run_l + G;                   // [G]

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      for (int i = 0; i < cnt; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES && !mbar_wait_bounded(empty + s, ((i / STAGES) - 1) & 1)) {
          flag_status(p.status, LOCKS_DEV_WAIT_TIMEOUT);
          break;
        }
        const int nv = s_nv[i], blk = s_blk[i];
        slot_nv[s] = nv;
        if (nv > 0) {
          const size_t off = (size_t(blk) * p.n_kv_heads + h) * (B * kHeadDim);
          const uint32_t bytes = uint32_t(nv) * kRowBytes;
          mbar_arrive_expect_tx(full + s, 2 * bytes);
          bulk_g2s(ring + size_t(s) * kSlotBytes, p.k_cache + off, bytes, full + s);
          bulk_g2s(ring + size_t(s) * kSlotBytes + kPageBytes, p.v_cache + off, bytes, full + s);
        } else {
          mbar_arrive(full + s);
        }
      }
    }
  } else {
    // ---------------- consumers ----------------
    const int dsub = lane & 7, tsub = lane >> 3;
    // query dims [8*dsub, 8*dsub+8) and [64+8*dsub, 64+8*dsub+8)
    float qf[G][16];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const __nv_bfloat16* qg = p.q + (size_t(b) * (p.n_kv_heads * G) + h * G + g) * kHeadDim;
      const uint4 a = *reinterpret_cast<const uint4*>(qg + 8 * dsub);
      const uint4 c = *reinterpret_cast<const uint4*>(qg + 64 + 8 * dsub);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        qf[g][2 * e] = bf16_lo(w[e]);
        qf[g][2 * e + 1] = bf16_hi(w[e]);
      }
    }
    if (lane < G) {
      run_m[lane] = -INFINITY;
      run_l[lane] = 0.f;
    }
    __syncwarp();

    constexpr int LPH = 32 / G;                                 // softmax lanes per head
    constexpr int TPL = LPH >= kTokPerWarp ? 1 : kTokPerWarp / LPH;
    const int hg = lane / LPH, li = lane % LPH;
    const int base = warp * kTokPerWarp;
    int done = cnt;
    bool aborted = false;
    for (int i = 0; i < cnt; ++i) {
      const int s = i % STAGES;
      if (!__all_sync(kFull, mbar_wait_bounded(full + s, (i / STAGES) & 1))) {
        if (lane == 0) flag_status(p.status, LOCKS_DEV_WAIT_TIMEOUT);
        aborted = true;
        done = i;
        break;
      }
      const int nv = slot_nv[s];
      if (nv > base) {
        const unsigned char* Ks = ring + size_t(s) * kSlotBytes;
        const unsigned char* Vs = Ks + kPageBytes;
        // ---- scores of this warp's 16 tokens ----
#pragma unroll
        for (int it = 0; it < kTokPerWarp / 4; ++it) {
          const int t = base + 4 * it + tsub;
          float part[G];
#pragma unroll
          for (int g = 0; g < G; ++g) part[g] = 0.f;
          if (t < nv) {
            const uint4 a = *reinterpret_cast<const uint4*>(Ks + t * kRowBytes + 16 * dsub);
            const uint4 c = *reinterpret_cast<const uint4*>(Ks + t * kRowBytes + 128 + 16 * dsub);
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float k0 = bf16_lo(w[e]), k1 = bf16_hi(w[e]);
#pragma unroll
              for (int g = 0; g < G; ++g) part[g] += qf[g][2 * e] * k0 + qf[g][2 * e + 1] * k1;
            }
          }
          TransposeReduce<G, 4>::run(part, lane);
          // lane holds head dsub / (8/G) (G <= 8) for token t
          constexpr int SG = G < 8 ? G : 8;
          if ((dsub & (8 / SG - 1)) == 0)
            s_buf[(dsub / (8 / SG)) * kTokPerWarp + 4 * it + tsub] = t < nv ? part[0] : -INFINITY;
        }
        __syncwarp();
        // ---- online softmax, head hg handled by lanes [hg*LPH, (hg+1)*LPH) ----
        {
          float sv[TPL];
          float mt = -INFINITY;
#pragma unroll
          for (int m = 0; m < TPL; ++m) {
            const int tl = li + LPH * m;
            sv[m] = tl < kTokPerWarp ? s_buf[hg * kTokPerWarp + tl] : -INFINITY;
            mt = fmaxf(mt, sv[m]);
          }
          mt = group_max<LPH>(mt);
          const float m_old = run_m[hg];
          const float m_new = fmaxf(m_old, mt);
          const float alpha = exp2f((m_old - m_new) * p.scale_log2);
          float ls = 0.f;
#pragma unroll
          for (int m = 0; m < TPL; ++m) {
            const int tl = li + LPH * m;
            const float pr = exp2f((sv[m] - m_new) * p.scale_log2);
            if (tl < kTokPerWarp) p_buf[tl * G + hg] = pr;
            ls += pr;
          }
          ls = group_sum<LPH>(ls);
          const float l_old = run_l[hg];
          __syncwarp();
          if (li == 0) {
            run_m[hg] = m_new;
            run_l[hg] = l_old * alpha + ls;
            alpha_buf[hg] = alpha;
          }
        }
        __syncwarp();
        // ---- acc = acc * alpha + P V over this warp's valid tokens ----
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float a = alpha_buf[g];
          acc[g][0] *= a; acc[g][1] *= a; acc[g][2] *= a; acc[g][3] *= a;
        }
        const int ntok = min(kTokPerWarp, nv - base);
        for (int tl = 0; tl < ntok; ++tl) {
          const float4 v = bf16x4_to_f4(
              *reinterpret_cast<const uint2*>(Vs + (base + tl) * kRowBytes + 8 * lane));
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float pr = p_buf[tl * G + g];
            acc[g][0] += pr * v.x; acc[g][1] += pr * v.y;
            acc[g][2] += pr * v.z; acc[g][3] += pr * v.w;
          }
        }
        __syncwarp();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
    }
    if (aborted) {
      for (int i = done; i < min(cnt, done + STAGES); ++i)
        mbar_wait_bounded(full + (i % STAGES), (i / STAGES) & 1);
    }
  }
  __syncthreads();

  // ---- merge the four warp states into the split's partial ----------------
  float* mbuf = reinterpret_cast<float*>(ring);    // [4][G][128], the ring is idle now
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int g = 0; g < G; ++g)
      *reinterpret_cast<float4*>(mbuf + (warp * G + g) * kHeadDim + 4 * lane) =
          make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
  }
  __syncthreads();
  const size_t part_stride = kPartStride;   // [m, l, pad, pad, acc[d]]: acc 16-byte aligned
  float* part = p.ws_part + (size_t(u) * p.n_splits_max + sp) * G * part_stride;
  for (int t = tid; t < G * 32; t += kDecThreads) {
    const int g = t >> 5, l4 = t & 31;
    float M = -INFINITY;
    for (int w = 0; w < kConsumerWarps; ++w)
      M = fmaxf(M, wbuf_all[w * warp_buf_floats<G>() + 2 * G * kTokPerWarp + g]);
    float L = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float* wbw = wbuf_all + w * warp_buf_floats<G>() + 2 * G * kTokPerWarp;
        const float f = exp2f((wbw[g] - M) * p.scale_log2);
        L += wbw[G + g] * f;
        const float4 a = *reinterpret_cast<const float4*>(mbuf + (w * G + g) * kHeadDim + 4 * l4);
        A.x += a.x * f; A.y += a.y * f; A.z += a.z * f; A.w += a.w * f;
      }
    }
    float* pg = part + g * part_stride;
    if (l4 == 0) { pg[0] = M; pg[1] = L; }
    *reinterpret_cast<float4*>(pg + 4 + 4 * l4) = A;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_is_last = (atomicAdd(p.ws_ticket + u, 1) == nsplits - 1);
  __syncthreads();
  if (!s_is_last) return;
  __threadfence();

  // ---- last split of the unit: merge every split -----------------------------
  // per-head maximum over the splits first (all loads in parallel) ...
  __shared__ float s_mmax[8];
  if (tid < G) s_mmax[tid] = -INFINITY;
  __syncthreads();
  for (int t = tid; t < nsplits * G; t += kDecThreads) {
    const int s2 = t / G, g = t % G;
    const float m2 = __ldcg(p.ws_part + ((size_t(u) * p.n_splits_max + s2) * G + g) * part_stride);
    if (m2 != -INFINITY) atomicMax_float(s_mmax + g, m2);
  }
  __syncthreads();
  // ... then the rescaled sums, whose loads no longer depend on each other
  for (int t = tid; t < G * 32; t += kDecThreads) {
    const int g = t >> 5, l4 = t & 31;
    const float M = s_mmax[g];
    float L = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll 8
      for (int s2 = 0; s2 < nsplits; ++s2) {
        const float* pg = p.ws_part + ((size_t(u) * p.n_splits_max + s2) * G + g) * part_stride;
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(pg));
        const float4 a2 = __ldcg(reinterpret_cast<const float4*>(pg + 4 + 4 * l4));
        const float f = ml.x == -INFINITY ? 0.f : exp2f((ml.x - M) * p.scale_log2);
        L += ml.y * f;
        A.x += a2.x * f; A.y += a2.y * f; A.z += a2.z * f; A.w += a2.w * f;
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* o = p.out + (size_t(b) * (p.n_kv_heads * G) + h * G + g) * kHeadDim + 4 * l4;
    const __nv_bfloat162 o01 = __floats2bfloat162_rn(A.x * inv, A.y * inv);
    const __nv_bfloat162 o23 = __floats2bfloat162_rn(A.z * inv, A.w * inv);
    uint2 ow;
    ow.x = *reinterpret_cast<const uint32_t*>(&o01);
    ow.y = *reinterpret_cast<const uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(o) = ow;
    if (l4 == 0 && p.out_lse)
      p.out_lse[size_t(b) * (p.n_kv_heads * G) + h * G + g] =
          L > 0.f ? M * p.scale + logf(L) : -INFINITY;
  }
  if (tid == 0) p.ws_ticket[u] = 0;
}

template <int G>
int launch_g(const DecodeParams& p, int gx, int gy, cudaStream_t stream) {
  constexpr int STAGES = 3;
  const size_t smem = size_t(STAGES) * kSlotBytes + 2 * STAGES * sizeof(uint64_t) +
                      ((STAGES + 3) / 4) * 4 * sizeof(int) +
                      kConsumerWarps * warp_buf_floats<G>() * sizeof(float);
  auto kern = decode_kernel<G, STAGES>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return LOCKS_ERR_CUDA;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(gx, gy);
  lc.blockDim = dim3(kDecThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kern, p) == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
}

}  // namespace

int launch_decode(const DecodeParams& p, int G, int gx, int gy, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_g<1>(p, gx, gy, stream);
    case 2: return launch_g<2>(p, gx, gy, stream);
    case 4: return launch_g<4>(p, gx, gy, stream);
    case 8: return launch_g<8>(p, gx, gy, stream);
    default: return LOCKS_ERR_UNSUPPORTED;
  }
}

}  // namespace locks
