// Parameter blocks and launchers shared between the C-ABI entry points
// (locks_api.cu) and the kernels.  Internal to the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/locks.h"

namespace locks {

constexpr size_t kMaxDynSmem = 227 * 1024;
// floats per (split, head) decode partial: m, l, two pad words, acc[head_dim]
constexpr int kPartStride = 4 + 128;

struct SelectParams {
  const __nv_bfloat16* q;        // [batch][H_q][d]
  const void* summaries;         // record pool
  const int32_t* block_table;    // [batch][max_pages]
  const int32_t* seq_lens;       // [batch]
  int32_t* selected;             // [batch][H_kv][k]
  float* page_lse;               // nullable [batch][H_q][max_pages]
  float* page_share;             // nullable [batch][H_kv][max_pages]
  int32_t* status;               // nullable
  float* ws_scores;              // [U][max_pages][G]
  float2* ws_part;               // [U][nseg_max][G] log-sum-exp partials
  uint2* ws_cand;                // [U][nslices_max][cand_per_slice] slice winners
  int32_t* ws_ticket;            // [U]
  size_t rec_bytes;
  int units, n_kv_heads, max_pages, num_blocks;
  int page_size;                 // tokens per page B (64 or 16)
  int k;                         // page budget
  int mc, per_cta, nseg_max;     // score kernel geometry (see select_geometry)
  int slice, nslices_max, fin_cap, cand_per_slice;
  float scale, scale_log2;
};

// Geometry of locks_select for a shape; the workspace size and the launch
// both come from here.
struct SelectGeom {
  int mc;            // candidate slots per unit (even)
  int per_cta;       // slots per score CTA (even)
  int n_score_ctas;
  int nseg_max;      // log-sum-exp partial slots per unit
  int slice;         // candidates per finalize CTA
  int nslices_max;
  int fin_cap;       // finalize shared-memory entries
  int cand_per_slice;
  size_t off_scores, off_part, off_cand, off_ticket, total;
};

struct DecodeParams {
  const __nv_bfloat16* q;        // [batch][H_q][d]
  const __nv_bfloat16* k_cache;  // [num_blocks][H_kv][B][d]
  const __nv_bfloat16* v_cache;
  const int32_t* block_table;    // [batch][max_pages]
  const int32_t* seq_lens;       // [batch]
  const int32_t* selected;       // nullable: [batch][H_kv][k]; NULL = every page
  __nv_bfloat16* out;            // [batch][H_q][d]
  float* out_lse;                // nullable [batch][H_q]
  int32_t* status;               // nullable
  float* ws_part;                // [U][n_splits_max][G][kPartStride]
  int32_t* ws_ticket;            // [U]
  int n_kv_heads, max_pages, num_blocks;
  int page_size;                 // tokens per page B (64 or 16)
  int k;                         // row stride of `selected`
  int pages_per_split, n_splits_max;
  float scale, scale_log2;
};

struct BuildParams {
  const __nv_bfloat16* k_cache;  // [num_blocks][H_kv][B][d]
  const int32_t* block_ids;      // [n_blocks]
  void* summaries;
  float* tail_energy;            // nullable [n_blocks][H_kv]
  int32_t* status;               // nullable [n_blocks][H_kv]
  size_t rec_bytes;
  int n_blocks, n_kv_heads, num_blocks, rank, max_sweeps;
  int skip_negative;             // a negative block id means "no page": skipped, not flagged
  int use_trd;                   // B = 64: tridiagonal top-r solver instead of Jacobi sweeps
};

struct AppendParams {
  const __nv_bfloat16* k_new;    // [batch][H_kv][d]
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_cache;        // [num_blocks][H_kv][B][d]
  __nv_bfloat16* v_cache;
  const int32_t* block_table;    // [batch][max_pages]
  int32_t* seq_lens;             // [batch], advanced by one
  int32_t* completed;            // nullable [batch]
  int32_t* status;               // nullable
  int n_kv_heads, max_pages, num_blocks, page_size;
};

// ctas_per_sm: score CTAs per SM the grid is sized for (see score_ctas_per_sm)
SelectGeom select_geometry(int units, int max_pages, int G, int k, int ctas_per_sm);
// Score CTAs per SM the grid is sized for.  Quantised records: 4, all
// resident at once (small records, denser arithmetic: more warps to hide
// instruction latency).  Float records: 2 resident per SM, in two waves, so
// that SMs that stream faster (HBM bandwidth per SM differs across the chip)
// take more of the second wave.
inline int score_ctas_per_sm(int /*summary_dtype*/) { return 4; }
// score kernel only, one definition per page size (locks_select.cu: 64,
// locks_score_b16.cu: 16)
int launch_score_b64(const SelectParams& p, int G, int RP, int dtype, int n_ctas,
                     cudaStream_t stream);
int launch_score_b16(const SelectParams& p, int G, int RP, int dtype, int n_ctas,
                     cudaStream_t stream);
int launch_select(const SelectParams& p, int G, int RP, int dtype, int n_score_ctas,
                  int n_slices, cudaStream_t stream);
int decode_pages_per_split(long units, int n_pages, int page_size);
int launch_decode(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int G,
                  int grid_x, int grid_y, cudaStream_t stream);
int launch_build(const BuildParams& p, int RP, int dtype, int page_size, cudaStream_t stream);
int launch_append(const AppendParams& p, int batch, cudaStream_t stream);

}  // namespace locks
