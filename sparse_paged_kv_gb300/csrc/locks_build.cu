// locks_build_summaries: the per-page spectral key summary of
// "Locks: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", section 4 "Build" (and the blog review's Algorithm 1).
//
// One CTA of 256 threads per (block, KV head) page, page size B = 64 or 16:
//   1. load the page's B bf16 keys, mu = mean of the keys, D = K - mu (fp32);
//   2. Gram A = D D^T (B x B), (B/16) x (B/16) register tiles per thread;
//   3. parallel cyclic Jacobi: each sweep is B-1 rounds of B/2 disjoint
//      (p, q) rotations (round-robin ordering, so every pair meets once per
//      sweep); a round applies A <- J^T A J as (B/2)^2 independent 2 x 2 block
//      transforms and U <- U J; sweeps stop when the off-diagonal Frobenius
//      norm falls below 1e-6 of the total (or at max_sweeps, flagged);
//   4. the top-r eigenpairs in descending order (ties: lower index); modes
//      with sigma^2 <= 1e-5 sigma_1^2 are dropped (zero basis column and
//      coefficients); V = D^T U_r S_r^-1, C = U_r S_r,
//      tau = sum of the remaining eigenvalues;
//   5. the record (mu, V, C) in the layout locks_select reads.
#include <cfloat>
#include <cstddef>
#include <type_traits>

#include "locks_common.cuh"
#include "locks_internal.h"

namespace locks {

namespace {

constexpr int kBuildThreads = 256;
constexpr int kDS = kHeadDim + 4;   // padded row stride of D (floats)
constexpr float kJacobiTol = 1e-6f;
constexpr float kDropRel = 1e-5f;

template <int PB>
struct BuildSmem {
  static constexpr int AS = PB + 1;   // padded row stride of A and U
  // D (the centred keys) is dead once the Gram sits in registers: A and U
  // reuse its space, and so does the quantised record's scratch (basis values
  // [16][d], then coefficient scales [B]), inside the dead A where it fits
  static constexpr int kScratch = 16 * kHeadDim + PB;
  static constexpr bool kScratchInA = PB * AS >= kScratch;
  static constexpr int kWorkD = PB * kDS;
  static constexpr int kWorkJ = 2 * PB * AS + (kScratchInA ? 0 : kScratch);
  float work[kWorkD > kWorkJ ? kWorkD : kWorkJ];
  float mu[kHeadDim];
  float4 rot[PB / 2];           // the round's rotations: c, s and the rows p, q (as bits)
  float red[kBuildThreads / 32 * 2];
  float lam[16];
  int order[16];
  float qscale[17];             // quantised record: column scales, then the centroid's
  float tau;
  int flag;
  unsigned char lp[PB - 1][PB / 2], lq[PB - 1][PB / 2];   // round labels (below)
  // the tridiagonal solver's scratch (B = 64 only)
  static constexpr int kTrd = PB == 64 ? 1 : 0;
  struct Trd {
    float d[PB], e[PB], e2[PB], tau[PB];  // T = Q^T A Q (diagonal, subdiagonal, its
                                          // squares); Householder scalars
    float v[PB], w[PB];                   // the current reflection's v and w
    float pp[4][PB];                      // partial products S v of the row groups
    float yc[PB][16], yz[PB][16];         // inverse iteration: the Thomas recurrences
    float sigma[16], lamr[16];            // shifts; Rayleigh quotients
    int clus[16];                         // cluster of each wanted eigenvalue
    float lo, hi, pivmin, tpiv, trace;
  } trd[kTrd];

  __device__ float* D() { return work; }             // [B][kDS]: steps 1-2
  __device__ float* A() { return work; }             // [B][AS]: steps 2-4
  __device__ float* U() { return work + PB * AS; }   // [B][AS]: steps 2-5
  __device__ float* Vs() { return work + (kScratchInA ? 0 : 2 * PB * AS); }   // step 5
  __device__ float* cs() { return Vs() + 16 * kHeadDim; }                       // step 5
};

// The rounds of the circle method on PB players (player PB-1 fixed, the other
// PB-1 rotate): pair 0 of round t is (t, PB-1), pair k > 0 is (t+k, t-k) mod
// PB-1. Which member of a pair is p and which q is free (a rotation is
// defined for either order), and it decides the shared-memory banks of the
// update: with a row stride of 1 mod 32, row x sits in bank x mod 32. Every
// residue class mod 32 holds two rows and every pair two members, so one
// member per pair can always be labelled p such that the 32 p rows (and so
// the 32 q rows) fall in distinct banks; lanes running over a round's pairs
// then touch 32 banks at once. The labels are found by walking the cycles
// that pairs and residue classes form (p = the smaller member when B <= 32,
// where all rows are in distinct banks anyway) and tabulated at compile time.
template <int PB>
struct alignas(16) RoundLabels {
  unsigned char p[PB - 1][PB / 2], q[PB - 1][PB / 2];
};

template <int PB>
constexpr RoundLabels<PB> make_round_labels() {
  constexpr int NPR = PB / 2;
  RoundLabels<PB> lab{};
  for (int t = 0; t < PB - 1; ++t) {
    int a[NPR] = {}, b[NPR] = {}, pair_of[PB] = {}, pick[NPR] = {};
    for (int k = 0; k < NPR; ++k) {
      a[k] = k == 0 ? t : (t + k) % (PB - 1);
      b[k] = k == 0 ? PB - 1 : (t - k + (PB - 1)) % (PB - 1);
      pair_of[a[k]] = k;
      pair_of[b[k]] = k;
      pick[k] = -1;
    }
    for (int k = 0; k < NPR; ++k) {
      if (pick[k] >= 0) continue;
      if (PB <= 32) {
        pick[k] = a[k] < b[k] ? a[k] : b[k];
        continue;
      }
      // label x as p; the other row of x's class must then be a q, so its
      // pair's other member is a p, and so on round the cycle
      int x = a[k], cur = k;
      for (;;) {
        pick[cur] = x;
        const int y = x ^ 32;
        const int j = pair_of[y];
        if (pick[j] >= 0) break;
        x = a[j] == y ? b[j] : a[j];
        cur = j;
      }
    }
    for (int k = 0; k < NPR; ++k) {
      lab.p[t][k] = static_cast<unsigned char>(pick[k]);
      lab.q[t][k] = static_cast<unsigned char>(pick[k] == a[k] ? b[k] : a[k]);
    }
  }
  return lab;
}

// every round pairs all rows (the circle method's pairs, each once) and, at
// B > 32, its p rows and its q rows each fall in 32 distinct banks
template <int PB>
constexpr bool round_labels_valid(const RoundLabels<PB>& lab) {
  for (int t = 0; t < PB - 1; ++t) {
    bool seen[PB] = {}, bank_p[32] = {}, bank_q[32] = {};
    for (int k = 0; k < PB / 2; ++k) {
      const int p = lab.p[t][k], q = lab.q[t][k];
      if (p >= PB || q >= PB || seen[p] || seen[q] || p == q) return false;
      seen[p] = seen[q] = true;
      const int a = k == 0 ? t : (t + k) % (PB - 1);
      const int b = k == 0 ? PB - 1 : (t - k + (PB - 1)) % (PB - 1);
      if (!((p == a && q == b) || (p == b && q == a))) return false;
      if (PB > 32) {
        if (bank_p[p % 32] || bank_q[q % 32]) return false;
        bank_p[p % 32] = bank_q[q % 32] = true;
      }
    }
  }
  return true;
}
static_assert(round_labels_valid<64>(make_round_labels<64>()), "round labels (B = 64)");
static_assert(round_labels_valid<16>(make_round_labels<16>()), "round labels (B = 16)");

__device__ const RoundLabels<64> kRoundLabels64 = make_round_labels<64>();
__device__ const RoundLabels<16> kRoundLabels16 = make_round_labels<16>();

template <int PB>
__device__ __forceinline__ const RoundLabels<PB>& round_labels() {
  if constexpr (PB == 64) return kRoundLabels64;
  else return kRoundLabels16;
}

// Quantised record (section 4 "Build": int4 basis with one scale per column,
// int8 coefficients and centroid with one scale per row): the float values
// the float record would hold, quantised symmetrically (scale = max|x| /
// qmax, code = round-half-even(x / scale), IEEE division, clamped), codes
// stored biased as in the layout of locks.h.
__device__ __forceinline__ uint32_t quant_biased(float x, float scale, int qmax) {
  if (!(scale > 0.f)) return uint32_t(qmax + 1);           // code 0
  const float c = fminf(fmaxf(rintf(__fdiv_rn(x, scale)), float(-qmax)), float(qmax));
  return uint32_t(int(c) + qmax + 1);
}

// v[k] = sum_i (key_i[t] - mu_t) U[i][order[k]] over the page's tokens: the
// unnormalised basis entries of dimension t for the modes k < r (modes past
// the rank read column 0 and are discarded by the caller).  The mode indices
// are read once; every token's row of U is a broadcast read.
template <int RP, int PB, int kAS, typename Smem>
__device__ __forceinline__ void basis_column_sums(const Smem& S, const __nv_bfloat16* kp, int t,
                                                  float mu_t, int r, float (&v)[RP]) {
  int ord[RP];
#pragma unroll
  for (int k = 0; k < RP; ++k) {
    ord[k] = k < r ? S.order[k] : 0;
    v[k] = 0.f;
  }
  const float* U = const_cast<Smem&>(S).U();
#pragma unroll 4
  for (int i = 0; i < PB; ++i) {
    const float dit = __bfloat162float(kp[i * kHeadDim + t]) - mu_t;
    const float* urow = U + i * kAS;
#pragma unroll
    for (int k = 0; k < RP; ++k) v[k] = fmaf(dit, urow[ord[k]], v[k]);
  }
}

template <int RP, int PB, typename Smem>
__device__ __forceinline__ void write_i4_record(Smem& S, const BuildParams& prm, int blk, int h,
                                                int r, const __nv_bfloat16* kp) {
  constexpr int kAS = Smem::AS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned char* rb = static_cast<unsigned char*>(prm.summaries) +
                      (size_t(blk) * prm.n_kv_heads + h) * prm.rec_bytes;
  const float* U = S.U();
  // basis values v_k[t] (as the float record stores them), D re-formed from
  // the key page kp as step 1 formed it
  float v[RP];
  if (tid < kHeadDim) basis_column_sums<RP, PB, kAS>(S, kp, tid, S.mu[tid], r, v);
  __syncthreads();
  float* Vs = S.Vs();                                      // [RP][d]
  if (tid < kHeadDim) {
#pragma unroll
    for (int k = 0; k < RP; ++k) {
      const float lam = k < r ? S.lam[k] : 0.f;
      Vs[k * kHeadDim + tid] = lam > 0.f ? v[k] * rsqrtf(lam) : 0.f;
    }
  }
  __syncthreads();
  // scales: basis column k (warp k % 8), the centroid (warp 0)
  for (int k = warp; k < RP; k += kBuildThreads / 32) {
    float am = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) am = fmaxf(am, fabsf(Vs[k * kHeadDim + lane + 32 * j]));
    am = group_max<32>(am);
    if (lane == 0) S.qscale[k] = am > 0.f ? __fdiv_rn(am, 7.f) : 0.f;
  }
  if (warp == 0) {
    float am = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) am = fmaxf(am, fabsf(S.mu[lane + 32 * j]));
    am = group_max<32>(am);
    if (lane == 0) S.qscale[16] = am > 0.f ? __fdiv_rn(am, 127.f) : 0.f;
  }
  __syncthreads();
  if (tid < RP * 16) {
    // basis word vq[k][t][j]: nibbles 0/4, 1/5 = k-step 2j at columns 2t/2t+1,
    // 2t+8/2t+9; nibbles 2/6, 3/7 = the same at k-step 2j+1 (see locks.h)
    const int k = tid >> 4, t = (tid >> 2) & 3, j = tid & 3;
    const float sc = S.qscale[k];
    const float* vk = Vs + k * kHeadDim;
    uint32_t w = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {                         // k-step 2j + h
      const int c0 = 16 * (2 * j + h) + 2 * t;
      w |= quant_biased(vk[c0], sc, 7) << (4 * (2 * h));
      w |= quant_biased(vk[c0 + 1], sc, 7) << (4 * (2 * h + 4));
      w |= quant_biased(vk[c0 + 8], sc, 7) << (4 * (2 * h + 1));
      w |= quant_biased(vk[c0 + 9], sc, 7) << (4 * (2 * h + 5));
    }
    reinterpret_cast<uint32_t*>(rb + i4_vq(RP))[tid] = w;
  }
  if (tid < RP) reinterpret_cast<float*>(rb)[tid] = S.qscale[tid];
  if (tid == RP) reinterpret_cast<float*>(rb)[RP] = S.qscale[16];
  if (tid >= 224) {
    // centroid word of lane l = 4g + t: columns 16g + 2t, +1, +8, +9
    const int l = tid - 224, g = l >> 2, t = l & 3;
    const float sc = S.qscale[16];
    const int c0 = 16 * g + 2 * t;
    const uint32_t w = quant_biased(S.mu[c0], sc, 127) | quant_biased(S.mu[c0 + 1], sc, 127) << 8 |
                       quant_biased(S.mu[c0 + 8], sc, 127) << 16 |
                       quant_biased(S.mu[c0 + 9], sc, 127) << 24;
    reinterpret_cast<uint32_t*>(rb + i4_mq(RP))[l] = w;
  }
  // coefficient rows: their scales first (one per token), then the codes in
  // the scorer's fragment order
  float* cs = S.cs();                                        // [PB]
  auto coeff = [&](int i, int k) {
    const float lam = k < r ? S.lam[k] : 0.f;
    return lam > 0.f ? U[i * kAS + S.order[k]] * sqrtf(lam) : 0.f;
  };
  if (tid < PB) {
    float am = 0.f;
#pragma unroll
    for (int k = 0; k < RP; ++k) am = fmaxf(am, fabsf(coeff(tid, k)));
    const float sc = am > 0.f ? __fdiv_rn(am, 127.f) : 0.f;
    cs[tid] = sc;
    reinterpret_cast<float*>(rb + i4_cscale(RP, PB))[tid] = sc;
  }
  __syncthreads();
  constexpr int KK = i4_kk(RP);
  for (int wi = tid; wi < (PB / 16) * KK * 32; wi += kBuildThreads) {
    const int m = wi / (KK * 32), kk = (wi / 32) % KK, l = wi % 32, g = l >> 2, t = l & 3;
    const int i0 = 16 * m + g, i1 = i0 + 8, k0 = 8 * kk + 2 * t;
    auto code = [&](int i, int k) {
      return k < RP ? quant_biased(coeff(i, k), cs[i], 127) : 128u;
    };
    const uint32_t w = code(i0, k0) | code(i0, k0 + 1) << 8 | code(i1, k0) << 16 |
                       code(i1, k0 + 1) << 24;
    reinterpret_cast<uint32_t*>(rb + i4_cq(RP))[wi] = w;
  }
}

// ---- top-r eigenpairs of the B x B Gram by tridiagonalisation (B = 64) ----
//   1. A = Q T Q^T, T tridiagonal, by B-2 Householder reflections (the
//      unblocked symmetric reduction: each step forms v from the column below
//      the diagonal, p = tau S v, w = p - (tau/2)(p.v) v and S -= v w^T + w v^T
//      on the trailing block S); v_k stays in A's column k below the diagonal;
//   2. the r largest eigenvalues of T, each bracketed by six rounds of
//      16-way multisection with Sturm counts (a half-warp per eigenvalue,
//      one count per lane): 24 bits of the Gershgorin interval;
//   3. their eigenvectors by two steps of inverse iteration with the bracket's
//      midpoint as shift (tridiagonal elimination, pivots kept off zero),
//      orthonormalised in order within clusters of equal eigenvalues; the
//      eigenvalues are then the Rayleigh quotients y^T T y;
//   4. U = Q Y by applying the reflections in reverse order.
// Leaves the eigenvectors as columns 0..r-1 of U (in descending eigenvalue
// order), lam[k] (0 for a dropped mode), order[k] = k and tau.
constexpr int kTrdRounds = 6;
constexpr int kTrdIters = 2;
constexpr float kTrdCluster = 1e-5f;   // relative gap below which eigenvalues are one cluster

__device__ __forceinline__ float trd_start(int i, int j) {
  // a fixed, data-independent start vector for inverse iteration
  uint32_t h = uint32_t(i) * 2654435761u + uint32_t(j) * 40503u + 12345u;
  h = (h ^ (h >> 15)) * 2246822519u;
  return float((h >> 8) & 0xffffu) * (1.f / 65536.f) - 0.5f;
}

template <int PB, typename Smem>
__device__ void trd_top_r(Smem& S, int r) {
  static_assert(PB == 64, "the tridiagonal solver is laid out for 64 x 64 Grams");
  constexpr int kAS = Smem::AS;
  constexpr int n = PB;
  auto& tr = S.trd[0];
  float* const A = S.A();
  float* const U = S.U();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- 1. Householder tridiagonalisation -----------------------------------
  // Every warp forms the step's reflection itself from the column below the
  // diagonal (no barrier between that and the matrix-vector product);
  // v_i = x_i / (x_0 - beta) is formed where it is used, and warp 0 stores
  // it in the column once the trailing block is updated.
  for (int k = 0; k < n - 2; ++k) {
    const int m = n - 1 - k;                  // rows k+1 .. n-1
    float* col = A + (k + 1) * kAS + k;       // col[i * kAS] = A[k+1+i][k]
    const float x0 = col[0];
    float sq = 0.f;
    for (int i = 1 + lane; i < m; i += 32) { const float x = col[i * kAS]; sq += x * x; }
    sq = group_sum<32>(sq);
    if (sq == 0.f) {                          // the column is already reduced
      if (tid == 0) { tr.tau[k] = 0.f; tr.e[k] = x0; }
      continue;                               // block-uniform: every warp saw the same column
    }
    const float beta = -copysignf(sqrtf(x0 * x0 + sq), x0);
    const float tau = (beta - x0) / beta;
    const float scale = 1.f / (x0 - beta);
    auto vv = [&](int i) { return i == 0 ? 1.f : col[i * kAS] * scale; };
    {
      // p = tau S v: thread (column i, row group g) sums rows j = g mod 4
      const int i = tid & (n - 1), g = tid >> 6;
      float acc = 0.f;
      if (i < m) {
#pragma unroll 4
        for (int j = g; j < m; j += 4) acc += A[(k + 1 + j) * kAS + k + 1 + i] * vv(j);
      }
      tr.pp[g][i] = acc;
      if (tid < m) tr.v[tid] = vv(tid);
    }
    __syncthreads();
    {
      // K = -(tau / 2) p.v (every warp), w = p + K v (rows 8 warp .. 8 warp + 7)
      float pv = 0.f;
      for (int i = lane; i < m; i += 32)
        pv += tau * (tr.pp[0][i] + tr.pp[1][i] + tr.pp[2][i] + tr.pp[3][i]) * tr.v[i];
      pv = group_sum<32>(pv);
      const float K = -0.5f * tau * pv;
      const int i = warp * (n / 8) + lane;
      if (lane < n / 8 && i < m)
        tr.w[i] = tau * (tr.pp[0][i] + tr.pp[1][i] + tr.pp[2][i] + tr.pp[3][i]) + K * tr.v[i];
    }
    __syncthreads();
    {
      // S -= v w^T + w v^T: thread column j, rows i = g mod 4
      const int j = tid & (n - 1);
      if (j < m) {
        const float vj = tr.v[j], wj = tr.w[j];
#pragma unroll 4
        for (int i = tid >> 6; i < m; i += 4)
          A[(k + 1 + i) * kAS + k + 1 + j] -= tr.v[i] * wj + tr.w[i] * vj;
      }
      // the reflection, kept in the reduced column for step 4
      if (warp == 0) {
        for (int i = 1 + lane; i < m; i += 32) col[i * kAS] = tr.v[i];
        if (lane == 0) { tr.tau[k] = tau; tr.e[k] = beta; }
      }
    }
    __syncthreads();
  }
  if (tid < n) tr.d[tid] = A[tid * kAS + tid];
  if (tid == 0) { tr.e[n - 2] = A[(n - 1) * kAS + n - 2]; tr.e[n - 1] = 0.f; }
  __syncthreads();

  // ---- 2. the r largest eigenvalues of T -------------------------------------
  if (warp == 0) {
    float lo = INFINITY, hi = -INFINITY, emax = 0.f, tr_sum = 0.f;
    for (int i = lane; i < n; i += 32) {
      const float ei = tr.e[i], em = i > 0 ? tr.e[i - 1] : 0.f;
      const float rad = fabsf(em) + fabsf(ei);
      lo = fminf(lo, tr.d[i] - rad);
      hi = fmaxf(hi, tr.d[i] + rad);
      emax = fmaxf(emax, ei * ei);
      tr_sum += tr.d[i];
      tr.e2[i] = ei * ei;
    }
    lo = -group_max<32>(-lo);
    hi = group_max<32>(hi);
    emax = group_max<32>(emax);
    tr_sum = group_sum<32>(tr_sum);
    if (lane == 0) {
      tr.lo = lo;
      tr.hi = hi;
      tr.pivmin = FLT_MIN * fmaxf(1.f, emax);
      tr.tpiv = fmaxf(FLT_MIN, 1.2e-7f * fmaxf(fabsf(lo), fabsf(hi)));
      tr.trace = tr_sum;
    }
  }
  __syncthreads();
  {
    // half-warp hw brackets eigenvalue hw from the top; lane hl counts the
    // eigenvalues below point hl + 1 of 16 (the points rise with hl, so the
    // lanes whose count is at most idx form a prefix)
    const int hw = tid >> 4, hl = tid & 15;
    if (2 * warp < r) {                       // both halves of the warp take part
      const int idx = n - 1 - min(hw, r - 1);
      const float pivmin = tr.pivmin;
      float a = tr.lo, b = tr.hi;
      for (int round = 0; round < kTrdRounds; ++round) {
        const float x = a + (b - a) * float(hl + 1) * (1.f / 16.f);
        float q = tr.d[0] - x;
        if (fabsf(q) < pivmin) q = -pivmin;
        int c = q < 0.f;
        for (int i = 1; i < n; ++i) {
          q = tr.d[i] - x - __fdividef(tr.e2[i - 1], q);
          if (fabsf(q) < pivmin) q = -pivmin;
          c += q < 0.f;
        }
        const unsigned le = (__ballot_sync(kFull, c <= idx) >> (lane & 16)) & 0xffffu;
        const int nle = __popc(le);
        const float a2 = a + (b - a) * float(nle) * (1.f / 16.f);
        const float b2 = a + (b - a) * float(nle + 1) * (1.f / 16.f);
        a = a2;
        b = b2;
      }
      if (hl == 0 && hw < r) tr.sigma[hw] = 0.5f * (a + b);
    }
  }
  __syncthreads();

  // ---- 3. eigenvectors of T by inverse iteration (warp 0, lane j) -----------
  if (warp == 0) {
    if (lane == 0) {
      const float tol = kTrdCluster * fmaxf(fabsf(tr.lo), fabsf(tr.hi));
      tr.clus[0] = 0;
      for (int j = 1; j < r; ++j) tr.clus[j] = (tr.sigma[j - 1] - tr.sigma[j]) < tol ? tr.clus[j - 1] : j;
    }
    if (lane < r)
      for (int i = 0; i < n; ++i) U[i * kAS + lane] = trd_start(i, lane);
    __syncwarp();
    const float tpiv = tr.tpiv;
    for (int it = 0; it < kTrdIters; ++it) {
      if (lane < r) {
        const int j = lane;
        const float sg = tr.sigma[j];
        float cp = 0.f, zp = 0.f;
        for (int i = 0; i < n; ++i) {
          const float em = i > 0 ? tr.e[i - 1] : 0.f;
          float piv = tr.d[i] - sg - em * cp;
          if (fabsf(piv) < tpiv) piv = piv < 0.f ? -tpiv : tpiv;
          const float inv = __fdividef(1.f, piv);
          cp = tr.e[i] * inv;
          zp = (U[i * kAS + j] - em * zp) * inv;
          tr.yc[i][j] = cp;
          tr.yz[i][j] = zp;
        }
        float x = tr.yz[n - 1][j], nrm = x * x;
        U[(n - 1) * kAS + j] = x;
        for (int i = n - 2; i >= 0; --i) {
          x = tr.yz[i][j] - tr.yc[i][j] * x;
          U[i * kAS + j] = x;
          nrm += x * x;
        }
        const bool ok = nrm > 0.f && nrm < INFINITY;
        const float sc = ok ? rsqrtf(nrm) : 0.f;
        for (int i = 0; i < n; ++i) U[i * kAS + j] = ok ? U[i * kAS + j] * sc : (i == j ? 1.f : 0.f);
      }
      __syncwarp();
      // Gram-Schmidt within clusters, in eigenvalue order (lanes over rows)
      for (int j = 1; j < r; ++j) {
        bool touched = false;
        for (int a = 0; a < j; ++a) {
          if (tr.clus[a] != tr.clus[j]) continue;
          float dt = U[lane * kAS + a] * U[lane * kAS + j] +
                     U[(lane + 32) * kAS + a] * U[(lane + 32) * kAS + j];
          dt = group_sum<32>(dt);
          U[lane * kAS + j] -= dt * U[lane * kAS + a];
          U[(lane + 32) * kAS + j] -= dt * U[(lane + 32) * kAS + a];
          touched = true;
          __syncwarp();
        }
        if (touched) {
          float nn = U[lane * kAS + j] * U[lane * kAS + j] +
                     U[(lane + 32) * kAS + j] * U[(lane + 32) * kAS + j];
          nn = group_sum<32>(nn);
          const float sc = nn > 0.f ? rsqrtf(nn) : 0.f;
          U[lane * kAS + j] *= sc;
          U[(lane + 32) * kAS + j] *= sc;
          __syncwarp();
        }
      }
    }
    // Rayleigh quotients y^T T y
    if (lane < r) {
      const int j = lane;
      float acc = 0.f;
      for (int i = 0; i < n; ++i) {
        const float yi = U[i * kAS + j];
        float t = tr.d[i] * yi;
        if (i > 0) t += tr.e[i - 1] * U[(i - 1) * kAS + j];
        if (i < n - 1) t += tr.e[i] * U[(i + 1) * kAS + j];
        acc += yi * t;
      }
      tr.lamr[j] = acc;
    }
    __syncwarp();
    if (lane == 0) {
      const float lam1 = tr.lamr[0];
      float top = 0.f;
      for (int k = 0; k < r; ++k) {
        const float lk = tr.lamr[k];
        top += lk;
        S.lam[k] = (lk > 0.f && lk > kDropRel * lam1) ? lk : 0.f;
        S.order[k] = k;
      }
      S.tau = fmaxf(0.f, tr.trace - top);
    }
  }
  __syncthreads();

  // ---- 4. U = Q Y: the reflections in reverse order (warp w, vectors w, w + 8)
  for (int j = warp; j < r; j += kBuildThreads / 32) {
    for (int k = n - 3; k >= 0; --k) {
      const float tau = tr.tau[k];
      if (tau == 0.f) continue;
      const int m = n - 1 - k;
      const float* col = A + (k + 1) * kAS + k;
      float s = 0.f;
      float v0 = 0.f, v1 = 0.f;
      if (lane < m) { v0 = lane == 0 ? 1.f : col[lane * kAS]; s += v0 * U[(k + 1 + lane) * kAS + j]; }
      if (lane + 32 < m) { v1 = col[(lane + 32) * kAS]; s += v1 * U[(k + 33 + lane) * kAS + j]; }
      s = tau * group_sum<32>(s);
      if (lane < m) U[(k + 1 + lane) * kAS + j] -= s * v0;
      if (lane + 32 < m) U[(k + 33 + lane) * kAS + j] -= s * v1;
      __syncwarp();
    }
  }
  __syncthreads();
}

// kTrd: top-r eigenpairs by the tridiagonal solver (trd_top_r) instead of
// cyclic Jacobi sweeps
template <int RP, typename T, int PB, bool kTrd>
__global__ void __launch_bounds__(kBuildThreads) build_kernel(const BuildParams prm) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BuildSmem<PB>& S = *reinterpret_cast<BuildSmem<PB>*>(smem_raw);
  float* const D = S.D();
  float* const A = S.A();
  float* const U = S.U();
  constexpr int kAS = BuildSmem<PB>::AS;
  constexpr int NPR = PB / 2;          // rotations per round
  constexpr int TT = PB / 16;          // Gram register tile edge
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pid = blockIdx.x;
  const int h = blockIdx.y;
  const int out_idx = pid * prm.n_kv_heads + h;
  const int blk = prm.block_ids[pid];
  if (blk < 0 || blk >= prm.num_blocks) {
    if (tid == 0 && prm.status)
      prm.status[out_idx] = (prm.skip_negative && blk < 0) ? 0 : LOCKS_DEV_BAD_BLOCK_ID << 16;
    return;
  }

  // ---- 1. keys -> D, mu ----------------------------------------------------
  const uint4* src = reinterpret_cast<const uint4*>(
      prm.k_cache + (size_t(blk) * prm.n_kv_heads + h) * (PB * kHeadDim));
#pragma unroll
  for (int e = 0; e < PB / 16; ++e) {
    const int idx = tid + kBuildThreads * e;       // 16-byte chunk of the 16 KiB page
    const int row = idx >> 4, col = (idx & 15) * 8;
    const uint4 w = src[idx];
    float* d = D + row * kDS + col;
    d[0] = bf16_lo(w.x); d[1] = bf16_hi(w.x); d[2] = bf16_lo(w.y); d[3] = bf16_hi(w.y);
    d[4] = bf16_lo(w.z); d[5] = bf16_hi(w.z); d[6] = bf16_lo(w.w); d[7] = bf16_hi(w.w);
  }
  __syncthreads();
  if (tid < kHeadDim) {
    float s = 0.f;
    for (int i = 0; i < PB; ++i) s += D[i * kDS + tid];
    S.mu[tid] = s * (1.f / PB);
  }
  __syncthreads();
  for (int idx = tid; idx < PB * kHeadDim; idx += kBuildThreads) {
    const int i = idx >> 7, t = idx & 127;
    D[i * kDS + t] -= S.mu[t];
  }
  __syncthreads();

  // ---- 2. Gram A = D D^T: thread (ti, tj) owns rows ti+16a, cols tj+16b ----
  {
    const int ti = tid >> 4, tj = tid & 15;
    float acc[TT][TT] = {};
    for (int c = 0; c < kHeadDim; c += 4) {
      float4 di[TT], dj[TT];
#pragma unroll
      for (int a = 0; a < TT; ++a) {
        di[a] = *reinterpret_cast<const float4*>(D + (ti + 16 * a) * kDS + c);
        dj[a] = *reinterpret_cast<const float4*>(D + (tj + 16 * a) * kDS + c);
      }
#pragma unroll
      for (int a = 0; a < TT; ++a)
#pragma unroll
        for (int bb = 0; bb < TT; ++bb)
          acc[a][bb] += di[a].x * dj[bb].x + di[a].y * dj[bb].y + di[a].z * dj[bb].z +
                        di[a].w * dj[bb].w;
    }
    __syncthreads();   // every read of D is done: A and U overwrite it
#pragma unroll
    for (int a = 0; a < TT; ++a)
#pragma unroll
      for (int bb = 0; bb < TT; ++bb) A[(ti + 16 * a) * kAS + tj + 16 * bb] = acc[a][bb];
  }
  for (int idx = tid; idx < PB * PB; idx += kBuildThreads) {
    const int i = idx / PB, j = idx % PB;
    U[i * kAS + j] = (i == j) ? 1.f : 0.f;
  }
  if constexpr (!kTrd) {
    static_assert(sizeof(RoundLabels<PB>) % 4 == 0 && offsetof(BuildSmem<PB>, lp) % 4 == 0 &&
                      offsetof(BuildSmem<PB>, lq) == offsetof(BuildSmem<PB>, lp) + sizeof(S.lp),
                  "round labels are copied as words");
    const uint32_t* src_l = reinterpret_cast<const uint32_t*>(&round_labels<PB>());
    uint32_t* dst_l = reinterpret_cast<uint32_t*>(&S.lp[0][0]);
    for (int w = tid; w < int(sizeof(RoundLabels<PB>) / 4); w += kBuildThreads) dst_l[w] = src_l[w];
  }
  __syncthreads();

  int sweeps = 0;
  bool converged = true;
  const int r = prm.rank;
  if constexpr (kTrd) {
    trd_top_r<PB>(S, r);
  } else {
    converged = false;
    // ---- 3. Jacobi sweeps ------------------------------------------------------
    for (;;) {
      // off-diagonal and total Frobenius norms
      float off = 0.f, tot = 0.f;
      for (int idx = tid; idx < PB * PB; idx += kBuildThreads) {
        const int i = idx / PB, j = idx % PB;
        const float a = A[i * kAS + j];
        tot += a * a;
        if (i != j) off += a * a;
      }
      off = group_sum<32>(off);
      tot = group_sum<32>(tot);
      if (lane == 0) { S.red[2 * warp] = off; S.red[2 * warp + 1] = tot; }
      __syncthreads();
      if (tid == 0) {
        float o = 0.f, t = 0.f;
        for (int w = 0; w < kBuildThreads / 32; ++w) { o += S.red[2 * w]; t += S.red[2 * w + 1]; }
        S.flag = (o <= kJacobiTol * kJacobiTol * t) ? 1 : 0;
      }
      __syncthreads();
      if (S.flag) { converged = true; break; }
      if (sweeps >= prm.max_sweeps) break;
      ++sweeps;
      for (int r = 0; r < PB - 1; ++r) {
        if (tid < NPR) {
          const int p = S.lp[r][tid], q = S.lq[r][tid];
          const float app = A[p * kAS + p], aqq = A[q * kAS + q], apq = A[p * kAS + q];
          float c = 1.f, s = 0.f;
          if (apq != 0.f) {
            const float theta = (aqq - app) / (2.f * apq);
            float t;
            if (fabsf(theta) > 1e18f) t = 0.5f / theta;
            else t = (theta >= 0.f ? 1.f : -1.f) / (fabsf(theta) + sqrtf(1.f + theta * theta));
            c = rsqrtf(1.f + t * t);
            s = t * c;
          }
          S.rot[tid] = make_float4(c, s, __int_as_float(p), __int_as_float(q));
        }
        __syncthreads();
        if (NPR * NPR >= kBuildThreads || tid < NPR * NPR) {
          // 2 x 2 blocks (K, L): rows (pK, qK), cols (pL, qL); B'' = J_K^T B J_L.
          // Block tid + 256 m is K = tid % NPR, L = (tid + 256 m) / NPR: the
          // lanes of a warp run over the pairs K, one column pair L per warp.
          static_assert(kBuildThreads % NPR == 0, "K is fixed per thread");
          const int K = tid % NPR;
          const float4 rK = S.rot[K];
          const float cK = rK.x, sK = rK.y;
          const int pK = __float_as_int(rK.z), qK = __float_as_int(rK.w);
  #pragma unroll
          for (int m = 0; m < (NPR * NPR + kBuildThreads - 1) / kBuildThreads; ++m) {
            const int L = (tid + kBuildThreads * m) / NPR;
            const float4 rL = S.rot[L];                 // one broadcast load per warp
            const float cL = rL.x, sL = rL.y;
            const int pL = __float_as_int(rL.z), qL = __float_as_int(rL.w);
            float* a00 = A + pK * kAS + pL;
            float* a01 = A + pK * kAS + qL;
            float* a10 = A + qK * kAS + pL;
            float* a11 = A + qK * kAS + qL;
            const float b00 = *a00, b01 = *a01, b10 = *a10, b11 = *a11;
            const float x00 = cK * b00 - sK * b10, x01 = cK * b01 - sK * b11;
            const float x10 = sK * b00 + cK * b10, x11 = sK * b01 + cK * b11;
            float n00 = x00 * cL - x01 * sL, n01 = x00 * sL + x01 * cL;
            float n10 = x10 * cL - x11 * sL, n11 = x10 * sL + x11 * cL;
            if (K == L) { n01 = 0.f; n10 = 0.f; }
            *a00 = n00; *a01 = n01; *a10 = n10; *a11 = n11;
          }
        }
        // U <- U J: item tid + 256 m is row i = item % B of pair L = item / B
        // (the lanes of a warp run over consecutive rows)
        if (NPR * PB >= kBuildThreads || tid < NPR * PB) {
  #pragma unroll
          for (int m = 0; m < (NPR * PB + kBuildThreads - 1) / kBuildThreads; ++m) {
            const int it = tid + kBuildThreads * m;
            const int i = it % PB, L = it / PB;
            const float4 rL = S.rot[L];
            const float cL = rL.x, sL = rL.y;
            const int pL = __float_as_int(rL.z), qL = __float_as_int(rL.w);
            const float up = U[i * kAS + pL], uq = U[i * kAS + qL];
            U[i * kAS + pL] = up * cL - uq * sL;
            U[i * kAS + qL] = up * sL + uq * cL;
          }
        }
        __syncthreads();
      }
    }

    // ---- 4. top-r eigenpairs (warp 0), tau ------------------------------------
    if (warp == 0) {
      // lane holds diagonal entries lane and lane + 32 (those past B count as taken)
      float v0 = lane < PB ? A[lane * kAS + lane] : 0.f;
      float v1 = lane + 32 < PB ? A[(lane + 32) * kAS + lane + 32] : 0.f;
      bool t0 = lane >= PB, t1 = lane + 32 >= PB;
      float lam1 = 0.f;
      for (int k = 0; k < r; ++k) {
        // candidate of this lane: larger value, ties -> lower index
        float bv = -INFINITY;
        int bi = 1 << 30;
        if (!t0) { bv = v0; bi = lane; }
        if (!t1 && (v1 > bv)) { bv = v1; bi = lane + 32; }
  #pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const float ov = __shfl_xor_sync(kFull, bv, o);
          const int oi = __shfl_xor_sync(kFull, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (bi == lane) t0 = true;
        if (bi == lane + 32) t1 = true;
        if (k == 0) lam1 = bv;
        if (lane == 0) {
          const bool keep = bv > 0.f && bv > kDropRel * lam1;
          S.lam[k] = keep ? bv : 0.f;
          S.order[k] = bi;
        }
      }
      float rest = (t0 ? 0.f : fmaxf(v0, 0.f)) + (t1 ? 0.f : fmaxf(v1, 0.f));
      rest = group_sum<32>(rest);
      if (lane == 0) S.tau = rest;
    }
    __syncthreads();
  }

  // ---- 5. record: W[0] = mu, W[1+k] = v_k, C[c][i][e] = u_ik sigma_k ----------
  // The basis V = D^T U_r S_r^-1 re-forms D from the key page: at B = 64 the
  // page is first brought back into the dead A (one coalesced round of loads
  // instead of one dependent load per token and dimension); at B = 16 it is
  // read where it is.
  const __nv_bfloat16* kp = prm.k_cache + (size_t(blk) * prm.n_kv_heads + h) * (PB * kHeadDim);
  if constexpr (PB == 64) {
    static_assert(PB * kHeadDim * 2 <= PB * BuildSmem<PB>::AS * 4, "the key page fits in A");
    uint4* dst = reinterpret_cast<uint4*>(A);
#pragma unroll
    for (int e = 0; e < PB / 16; ++e) dst[tid + kBuildThreads * e] = src[tid + kBuildThreads * e];
    __syncthreads();
    kp = reinterpret_cast<const __nv_bfloat16*>(A);
  }
  if constexpr (std::is_same_v<T, I4Rec>) {
    write_i4_record<RP, PB>(S, prm, blk, h, r, kp);
  } else {
    T* rec = reinterpret_cast<T*>(static_cast<unsigned char*>(prm.summaries) +
                                  (size_t(blk) * prm.n_kv_heads + h) * prm.rec_bytes);
    if (tid < kHeadDim) {
      const int t = tid;
      const float mu_t = S.mu[t];
      st_elem(rec + t, mu_t);
      // D re-formed from the key page as step 1 formed it (A and U hold its space)
      float v[RP];
      basis_column_sums<RP, PB, kAS>(S, kp, t, mu_t, r, v);
#pragma unroll
      for (int k = 0; k < RP; ++k) {
        const float lam = k < r ? S.lam[k] : 0.f;
        st_elem(rec + (1 + k) * kHeadDim + t, lam > 0.f ? v[k] * rsqrtf(lam) : 0.f);
      }
    } else {
      T* C = rec + rec_w_elems(RP);
      for (int idx = tid - kHeadDim; idx < PB * RP; idx += kBuildThreads - kHeadDim) {
        const int i = idx / RP, k = idx % RP;
        const float lam = k < r ? S.lam[k] : 0.f;
        const float c = lam > 0.f ? U[i * kAS + S.order[k]] * sqrtf(lam) : 0.f;
        st_elem(C + ((k >> 2) * PB + i) * 4 + (k & 3), c);
      }
    }
  }
  if (tid == 0) {
    if (prm.tail_energy) prm.tail_energy[out_idx] = S.tau;
    if (prm.status) prm.status[out_idx] = sweeps | (converged ? 0 : (LOCKS_DEV_NOT_CONVERGED << 16));
  }
}

template <int RP, typename T, int PB>
int launch_t(const BuildParams& p, cudaStream_t stream) {
  const size_t smem = sizeof(BuildSmem<PB>);
  auto kern = (PB == 64 && p.use_trd) ? build_kernel<RP, T, PB, PB == 64>
                                      : build_kernel<RP, T, PB, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return LOCKS_ERR_CUDA;
  kern<<<dim3(p.n_blocks, p.n_kv_heads), kBuildThreads, smem, stream>>>(p);
  return cudaPeekAtLastError() == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
}

template <int PB, typename T>
int launch_rp(const BuildParams& p, int RP, cudaStream_t stream) {
  switch (RP) {
    case 4: return launch_t<4, T, PB>(p, stream);
    case 8: return launch_t<8, T, PB>(p, stream);
    case 16: return launch_t<16, T, PB>(p, stream);
    default: return LOCKS_ERR_UNSUPPORTED;
  }
}

template <int PB>
int launch_pb(const BuildParams& p, int RP, int dtype, cudaStream_t stream) {
  if (dtype == LOCKS_SUMMARY_F32) return launch_rp<PB, float>(p, RP, stream);
  if (dtype == LOCKS_SUMMARY_BF16) return launch_rp<PB, __nv_bfloat16>(p, RP, stream);
  if (dtype == LOCKS_SUMMARY_I4) return launch_rp<PB, I4Rec>(p, RP, stream);
  return LOCKS_ERR_UNSUPPORTED;
}

}  // namespace

int launch_build(const BuildParams& p, int RP, int dtype, int page_size, cudaStream_t stream) {
  if (page_size == 64) return launch_pb<64>(p, RP, dtype, stream);
  if (page_size == 16) return launch_pb<16>(p, RP, dtype, stream);
  return LOCKS_ERR_UNSUPPORTED;
}

}  // namespace locks
