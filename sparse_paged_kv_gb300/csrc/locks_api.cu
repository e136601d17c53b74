// C-ABI entry points of libsparse_paged_kv (declared in include/locks.h):
// argument validation, workspace sizing and kernel dispatch.  Nothing here
// allocates, frees or synchronises.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "locks_common.cuh"
#include "locks_internal.h"

namespace {

using locks::kHeadDim;

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool is_pow2_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

int check_cfg(const locks_cfg_t* c) {
  if (!c) return LOCKS_ERR_INVALID_ARG;
  if (c->batch < 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->max_pages <= 0 ||
      c->num_blocks <= 0 || c->rank <= 0 || c->head_dim <= 0 || c->page_size <= 0)
    return LOCKS_ERR_INVALID_ARG;
  if (c->n_q_heads % c->n_kv_heads != 0) return LOCKS_ERR_INVALID_ARG;
  if (c->summary_dtype != LOCKS_SUMMARY_F32 && c->summary_dtype != LOCKS_SUMMARY_BF16 &&
      c->summary_dtype != LOCKS_SUMMARY_I4)
    return LOCKS_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim || (c->page_size != 64 && c->page_size != 16))
    return LOCKS_ERR_UNSUPPORTED;
  if (c->rank > 16) return LOCKS_ERR_UNSUPPORTED;
  // the score kernel keeps a record index in an int and a page index in 24 bits
  if (c->max_pages >= (1 << 24) || int64_t(c->num_blocks) * c->n_kv_heads >= (int64_t(1) << 31))
    return LOCKS_ERR_UNSUPPORTED;
  if (!is_pow2_group(c->n_q_heads / c->n_kv_heads)) return LOCKS_ERR_UNSUPPORTED;
  return LOCKS_OK;
}

int group_of(const locks_cfg_t* c) { return c->n_q_heads / c->n_kv_heads; }

size_t elem_bytes(const locks_cfg_t* c) { return c->summary_dtype == LOCKS_SUMMARY_F32 ? 4 : 2; }

int page_budget(int budget_tokens, int page_size) {
  return (budget_tokens + page_size - 1) / page_size;   // k = ceil(b / B)
}

// ---- decode workspace -------------------------------------------------------
struct DecodeLayout {
  size_t part, ticket, total;
  int pages_per_split, n_splits_max;
};

DecodeLayout decode_layout(const locks_cfg_t* c, int n_pages) {
  DecodeLayout L;
  const int G = group_of(c);
  const size_t U = size_t(c->batch) * c->n_kv_heads;
  L.pages_per_split = locks::decode_pages_per_split(long(U), n_pages, c->page_size);
  L.n_splits_max = n_pages > 0 ? (n_pages + L.pages_per_split - 1) / L.pages_per_split : 1;
  L.part = 0;
  L.ticket = align_up(U * L.n_splits_max * G * locks::kPartStride * sizeof(float));
  L.total = L.ticket + align_up(U * sizeof(int32_t));
  return L;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A KV pool viewed as a 2-D bf16 tensor of (num_blocks * n_kv_heads * B) rows
// of head_dim elements, read in boxes of B rows x 64 columns (one page-head's
// half rows) with 128-byte swizzle.
bool encode_pool_map(CUtensorMap* m, const void* pool, const locks_cfg_t* c) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cuuint64_t(c->head_dim),
                              cuuint64_t(c->num_blocks) * c->n_kv_heads * c->page_size};
  const cuuint64_t strides[1] = {cuuint64_t(c->head_dim) * 2};
  const cuuint32_t box[2] = {64, cuuint32_t(c->page_size)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int decode_common(const locks_cfg_t* cfg, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_table, const int32_t* seq_lens, const int32_t* selected,
                  int32_t k, int n_list_max, void* out, float* out_lse, void* workspace,
                  size_t workspace_bytes, int32_t* status, void* stream) {
  int rc = check_cfg(cfg);
  if (rc != LOCKS_OK) return rc;
  if (cfg->batch == 0) return LOCKS_OK;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !workspace)
    return LOCKS_ERR_INVALID_ARG;
  const DecodeLayout L = decode_layout(cfg, n_list_max);
  if (workspace_bytes < L.total) return LOCKS_ERR_WORKSPACE;
  locks::DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  p.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.selected = selected;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.out_lse = out_lse;
  p.status = status;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.ws_part = reinterpret_cast<float*>(ws + L.part);
  p.ws_ticket = reinterpret_cast<int32_t*>(ws + L.ticket);
  p.n_kv_heads = cfg->n_kv_heads;
  p.max_pages = cfg->max_pages;
  p.num_blocks = cfg->num_blocks;
  p.page_size = cfg->page_size;
  p.k = k;
  p.pages_per_split = L.pages_per_split;
  p.n_splits_max = L.n_splits_max;
  p.scale = float(1.0 / std::sqrt(double(cfg->head_dim)));
  p.scale_log2 = float(1.4426950408889634 / std::sqrt(double(cfg->head_dim)));
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return LOCKS_ERR_INVALID_ARG;                     // tensor maps need 16-byte bases
  CUtensorMap tk, tv;
  if (!encode_pool_map(&tk, k_cache, cfg) || !encode_pool_map(&tv, v_cache, cfg))
    return LOCKS_ERR_CUDA;
  const int U = cfg->batch * cfg->n_kv_heads;
  return locks::launch_decode(p, tk, tv, group_of(cfg), L.n_splits_max, U,
                              static_cast<cudaStream_t>(stream));
}

}  // namespace

namespace {

int build_common(const locks_cfg_t* cfg, const void* k_cache, const int32_t* block_ids,
                 int32_t n_blocks, void* summaries, float* tail_energy, int32_t* status,
                 int32_t max_sweeps, int skip_negative, void* stream) {
  int rc = check_cfg(cfg);
  if (rc != LOCKS_OK) return rc;
  if (n_blocks < 0 || max_sweeps < 0) return LOCKS_ERR_INVALID_ARG;
  if (n_blocks == 0) return LOCKS_OK;
  if (!k_cache || !block_ids || !summaries) return LOCKS_ERR_INVALID_ARG;
  locks::BuildParams p;
  p.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  p.block_ids = block_ids;
  p.summaries = summaries;
  p.tail_energy = tail_energy;
  p.status = status;
  p.rec_bytes = locks_summary_record_bytes(cfg);
  p.n_blocks = n_blocks;
  p.n_kv_heads = cfg->n_kv_heads;
  p.num_blocks = cfg->num_blocks;
  p.rank = cfg->rank;
  p.max_sweeps = max_sweeps == 0 ? 20 : max_sweeps;
  p.use_trd = max_sweeps == 0 && cfg->page_size == 64;   // a sweep cap asks for Jacobi
  p.skip_negative = skip_negative;
  return locks::launch_build(p, locks::rank_cap(cfg->rank), cfg->summary_dtype, cfg->page_size,
                             static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

size_t locks_summary_record_bytes(const locks_cfg_t* cfg) {
  if (check_cfg(cfg) != LOCKS_OK) return 0;
  const int rp = locks::rank_cap(cfg->rank);
  if (cfg->summary_dtype == LOCKS_SUMMARY_I4) return size_t(locks::i4_bytes(rp, cfg->page_size));
  return size_t(locks::rec_elems(rp, cfg->page_size)) * elem_bytes(cfg);
}

size_t locks_summary_bytes(const locks_cfg_t* cfg) { return locks_summary_record_bytes(cfg); }

size_t locks_select_workspace_bytes(const locks_cfg_t* cfg, int32_t budget_tokens) {
  if (check_cfg(cfg) != LOCKS_OK) return 0;
  const int k = page_budget(budget_tokens, cfg->page_size);
  if (budget_tokens <= 0 || k < 2) return 0;
  if (cfg->batch == 0) return 0;
  return locks::select_geometry(cfg->batch * cfg->n_kv_heads, cfg->max_pages, group_of(cfg), k,
                                locks::score_ctas_per_sm(cfg->summary_dtype))
      .total;
}

size_t locks_decode_workspace_bytes(const locks_cfg_t* cfg, int32_t n_pages) {
  if (check_cfg(cfg) != LOCKS_OK || n_pages < 0) return 0;
  return decode_layout(cfg, n_pages).total;
}

int locks_build_summaries(const locks_cfg_t* cfg, const void* k_cache, const int32_t* block_ids,
                          int32_t n_blocks, void* summaries, float* tail_energy, int32_t* status,
                          int32_t max_sweeps, void* stream) {
  return build_common(cfg, k_cache, block_ids, n_blocks, summaries, tail_energy, status,
                      max_sweeps, 0, stream);
}

int locks_build_completed(const locks_cfg_t* cfg, const void* k_cache, const int32_t* completed,
                          int32_t n, void* summaries, float* tail_energy, int32_t* status,
                          int32_t max_sweeps, void* stream) {
  return build_common(cfg, k_cache, completed, n, summaries, tail_energy, status, max_sweeps, 1,
                      stream);
}

int locks_append_kv(const locks_cfg_t* cfg, const void* k_new, const void* v_new, void* k_cache,
                    void* v_cache, const int32_t* block_table, int32_t* seq_lens,
                    int32_t* completed, int32_t* status, void* stream) {
  int rc = check_cfg(cfg);
  if (rc != LOCKS_OK) return rc;
  if (cfg->batch == 0) return LOCKS_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens)
    return LOCKS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
       reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return LOCKS_ERR_INVALID_ARG;                     // rows move as 16-byte words
  locks::AppendParams p;
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  p.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.completed = completed;
  p.status = status;
  p.n_kv_heads = cfg->n_kv_heads;
  p.max_pages = cfg->max_pages;
  p.num_blocks = cfg->num_blocks;
  p.page_size = cfg->page_size;
  return locks::launch_append(p, cfg->batch, static_cast<cudaStream_t>(stream));
}

int locks_select(const locks_cfg_t* cfg, const void* q, const void* summaries,
                 const int32_t* block_table, const int32_t* seq_lens, int32_t budget_tokens,
                 int32_t* selected, float* page_lse, float* page_share, void* workspace,
                 size_t workspace_bytes, int32_t* status, void* stream) {
  int rc = check_cfg(cfg);
  if (rc != LOCKS_OK) return rc;
  const int k = page_budget(budget_tokens, cfg->page_size);
  if (budget_tokens <= 0 || k < 2) return LOCKS_ERR_INVALID_ARG;
  if (k > 256) return LOCKS_ERR_UNSUPPORTED;
  if (cfg->batch == 0) return LOCKS_OK;
  if (!q || !summaries || !block_table || !seq_lens || !selected || !workspace)
    return LOCKS_ERR_INVALID_ARG;
  const int U = cfg->batch * cfg->n_kv_heads;
  const locks::SelectGeom L = locks::select_geometry(U, cfg->max_pages, group_of(cfg), k,
                                                     locks::score_ctas_per_sm(cfg->summary_dtype));
  if (workspace_bytes < L.total) return LOCKS_ERR_WORKSPACE;
  locks::SelectParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.summaries = summaries;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.selected = selected;
  p.page_lse = page_lse;
  p.page_share = page_share;
  p.status = status;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.ws_scores = reinterpret_cast<float*>(ws + L.off_scores);
  p.ws_part = reinterpret_cast<float2*>(ws + L.off_part);
  p.ws_cand = reinterpret_cast<uint2*>(ws + L.off_cand);
  p.ws_ticket = reinterpret_cast<int32_t*>(ws + L.off_ticket);
  p.rec_bytes = locks_summary_record_bytes(cfg);
  p.units = U;
  p.n_kv_heads = cfg->n_kv_heads;
  p.max_pages = cfg->max_pages;
  p.num_blocks = cfg->num_blocks;
  p.page_size = cfg->page_size;
  p.k = k;
  p.mc = L.mc;
  p.per_cta = L.per_cta;
  p.nseg_max = L.nseg_max;
  p.slice = L.slice;
  p.nslices_max = L.nslices_max;
  p.fin_cap = L.fin_cap;
  p.cand_per_slice = L.cand_per_slice;
  p.scale = float(1.0 / std::sqrt(double(cfg->head_dim)));
  p.scale_log2 = float(1.4426950408889634 / std::sqrt(double(cfg->head_dim)));
  return locks::launch_select(p, group_of(cfg), locks::rank_cap(cfg->rank), cfg->summary_dtype,
                              L.n_score_ctas, L.nslices_max, static_cast<cudaStream_t>(stream));
}

int locks_sparse_decode(const locks_cfg_t* cfg, const void* q, const void* k_cache,
                        const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                        const int32_t* selected, int32_t k, void* out, float* out_lse,
                        void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  if (!cfg || !selected || k <= 0) return LOCKS_ERR_INVALID_ARG;
  return decode_common(cfg, q, k_cache, v_cache, block_table, seq_lens, selected, k, k, out,
                       out_lse, workspace, workspace_bytes, status, stream);
}

int locks_dense_decode(const locks_cfg_t* cfg, const void* q, const void* k_cache,
                       const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                       void* out, float* out_lse, void* workspace, size_t workspace_bytes,
                       int32_t* status, void* stream) {
  if (!cfg) return LOCKS_ERR_INVALID_ARG;
  return decode_common(cfg, q, k_cache, v_cache, block_table, seq_lens, nullptr, 0,
                       cfg->max_pages, out, out_lse, workspace, workspace_bytes, status, stream);
}

const char* locks_status_string(int code) {
  switch (code) {
    case LOCKS_OK: return "ok";
    case LOCKS_ERR_INVALID_ARG: return "invalid argument";
    case LOCKS_ERR_UNSUPPORTED: return "unsupported shape";
    case LOCKS_ERR_WORKSPACE: return "workspace too small";
    case LOCKS_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

int locks_abi_version(void) { return LOCKS_ABI_VERSION; }

}  // extern "C"
