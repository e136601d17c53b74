// locks_append_kv: the cache write of a decode step.  Each sequence's newest
// token (its key and value rows for every KV head) goes to position
// seq_lens[b] of the paged pools, the sequence length advances by one, and the
// physical block of a page the token completes is reported, so that its
// summary can be built right away ("Locks: Page-Local Compact Key Summaries
// for Efficient Long-Context Decoding", section 4 "Build": a page is
// summarised once, when it completes).
//
// One CTA per sequence: thread 0 reads the length and the block-table entry,
// then the CTA copies 2 x H_kv rows of 256 bytes as 16-byte words.
#include "locks_common.cuh"
#include "locks_internal.h"

namespace locks {

namespace {

constexpr int kAppendThreads = 256;
constexpr int kRowWords = kHeadDim * 2 / 16;   // 16-byte words of one bf16 row

__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendParams p) {
  // the selection's score kernel that follows may start launching at once:
  // it reads nothing before its own wait for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x;
  const int B = p.page_size;
  __shared__ int s_blk, s_pos;
  if (threadIdx.x == 0) {
    const int t = p.seq_lens[b];
    int blk = -1;
    if (t < 0 || t >= p.max_pages * B) {
      flag_status(p.status, LOCKS_DEV_BAD_SEQ_LEN);
    } else {
      blk = p.block_table[size_t(b) * p.max_pages + t / B];
      if (blk < 0 || blk >= p.num_blocks) {
        flag_status(p.status, LOCKS_DEV_BAD_BLOCK_ID);
        blk = -1;
      }
    }
    s_blk = blk;
    s_pos = t;
  }
  __syncthreads();
  const int blk = s_blk, pos = s_pos;
  if (blk >= 0) {
    const int slot = pos % B;
    const int n_words = 2 * p.n_kv_heads * kRowWords;
    for (int i = threadIdx.x; i < n_words; i += kAppendThreads) {
      const int kv = i / (p.n_kv_heads * kRowWords);
      const int h = (i / kRowWords) % p.n_kv_heads, c = i % kRowWords;
      const uint4* src = reinterpret_cast<const uint4*>(kv ? p.v_new : p.k_new) +
                         (size_t(b) * p.n_kv_heads + h) * kRowWords + c;
      uint4* dst = reinterpret_cast<uint4*>(kv ? p.v_cache : p.k_cache) +
                   ((size_t(blk) * p.n_kv_heads + h) * B + slot) * kRowWords + c;
      *dst = __ldg(src);
    }
  }
  if (threadIdx.x == 0) {
    if (blk >= 0) p.seq_lens[b] = pos + 1;
    if (p.completed) p.completed[b] = (blk >= 0 && (pos + 1) % B == 0) ? blk : -1;
  }
}

}  // namespace

int launch_append(const AppendParams& p, int batch, cudaStream_t stream) {
  append_kernel<<<batch, kAppendThreads, 0, stream>>>(p);
  return cudaPeekAtLastError() == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
}

}  // namespace locks
