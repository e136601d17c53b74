// locks_select_noalloc: locks_select without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they select
// pages: code running inside a memory pool or arena that owns every byte of
// the GPU (a serving engine that has handed its whole KV budget to a cache
// allocator), plugins whose host framework forbids cudaMalloc on its hot path
// because it would synchronise the device or fragment the pool, and embedded
// callers that have no allocator at all.  For them this entry point keeps the
// selection scratch (per-page scores, per-chunk log-sum-exp partials and the
// completion tickets) in one fixed, file-scope device array instead.
//
// The array costs LOCKS_SELECT_NOALLOC_MAX_BYTES of device memory on every GPU
// that loads the library, held until the process exits.  Its device address is
// looked up once per device context: on the first call made while that device
// is current, and again on the first call after the context was destroyed and
// created anew (cudaDeviceReset reloads the library's module, which can move
// the array).  Those calls should therefore come before any stream capture.
// Every call clears the part of the array it uses (an asynchronous memset on
// the caller's stream) and then runs the same selection kernel as
// locks_select.  All calls share the one array: calls that may overlap on the
// GPU (different streams without ordering between them) race on it.
#include <array>
#include <mutex>

#include "locks_common.cuh"
#include "locks_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_select_scratch[LOCKS_SELECT_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
struct ScratchSlot {
  unsigned long long ctx_id;   // cuCtxGetId of the context the address belongs to
  void* ptr;                   // device address of g_select_scratch in that context
};
std::array<ScratchSlot, kMaxDevices> g_scratch{};   // per device ordinal

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The id of the calling thread's current context (unique within the process
// and never reused, unlike the context handle); false when no context is
// current or the driver does not offer the calls.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's context, looked
// up again whenever that context is not the one the cached address came from.
int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LOCKS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchSlot& slot = g_scratch[dev];
  unsigned long long id = 0;
  if (slot.ptr == nullptr || !current_context_id(&id) || id != slot.ctx_id) {
    void* p = nullptr;   // the lookup also makes the device's primary context current
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || p == nullptr)
      return LOCKS_ERR_CUDA;
    if (!current_context_id(&id)) return LOCKS_ERR_CUDA;
    slot.ctx_id = id;
    slot.ptr = p;
  }
  *out = slot.ptr;
  return LOCKS_OK;
}

}  // namespace

extern "C" int locks_select_noalloc(const locks_cfg_t* cfg, const void* q, const void* summaries,
                                    const int32_t* block_table, const int32_t* seq_lens,
                                    int32_t budget_tokens, int32_t* selected, float* page_lse,
                                    float* page_share, int32_t* status, void* stream) {
  if (!cfg) return LOCKS_ERR_INVALID_ARG;
  // bytes of scratch this shape needs (0 when the shape is invalid; locks_select
  // then reports why)
  const size_t need = locks_select_workspace_bytes(cfg, budget_tokens);
  if (need > LOCKS_SELECT_NOALLOC_MAX_BYTES) return LOCKS_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != LOCKS_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (need > 0 && cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) return LOCKS_ERR_CUDA;
  return locks_select(cfg, q, summaries, block_table, seq_lens, budget_tokens, selected, page_lse,
                      page_share, scratch, LOCKS_SELECT_NOALLOC_MAX_BYTES, status, stream);
}
