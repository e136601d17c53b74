/*
 * locks.h -- C ABI of the Locks decode-attention hot path on one GB300 (sm_103a).
 *
 * The method is the one of "Locks: Page-Local Compact Key Summaries for
 * Efficient Long-Context Decoding" (arXiv 2607.24555): every completed page of
 * a paged KV cache gets its own rank-r spectral key summary (section 4,
 * "Build"); each decode step scores every candidate page by the log-sum-exp of
 * its reconstructed within-page logits (section 4, Eq. (1)), normalises the
 * scores into per-head page-mass shares, averages the shares over the GQA
 * group, keeps the sink page and the most recent page and the top-(k-2)
 * remaining pages under the token budget (section 2; section 4; Cor. 3), and
 * attends only the selected pages.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All pointers named *_cache, q, summaries, block_table, seq_lens, selected,
 *    out*, page_*, workspace, status, tail_energy and block_ids are DEVICE
 *    pointers owned by the caller.  The library never allocates, frees or
 *    synchronises; every call only enqueues kernels on `stream` (a
 *    cudaStream_t passed as void*, NULL = legacy default stream).
 *  - The return value reports argument validation and launch errors only
 *    (LOCKS_ERR_*).  Conditions found on the device (a block id outside the
 *    pool, a page id outside the sequence, a bounded wait that ran out, a
 *    Jacobi solve that did not converge) are OR-ed as LOCKS_DEV_* bits into the
 *    caller's `status` word(s) when that pointer is non-NULL; the offending
 *    page is skipped.  Read them after synchronising the stream.
 *  - bf16 is IEEE bfloat16 stored as 16-bit words.
 *  - KV pools are [num_blocks][n_kv_heads][page_size][head_dim] bf16: each
 *    (block, KV head) page is contiguous.  Logical page j of sequence b lives
 *    in physical block block_table[b * max_pages + j].  Only the first
 *    seq_lens[b] tokens of a sequence are ever read; the rest of its tail page
 *    may hold anything (NaN included).
 *  - Query head h uses KV head h / G, with G = n_q_heads / n_kv_heads
 *    (contiguous grouping).  Logits are scaled by 1/sqrt(head_dim)
 *    (section 2).
 *  - Calls that use a workspace require it to be zero-filled before its first
 *    use (cudaMemset once); every call leaves it ready for the next call, so
 *    the same workspace can be replayed inside a CUDA graph.  Calls that share
 *    a workspace must not overlap on the GPU.
 *
 * Supported shapes: head_dim = 128; page_size = 64 or 16; 1 <= rank <= 16;
 * G in {1, 2, 4, 8}; max_pages < 2^24; num_blocks * n_kv_heads < 2^31.
 * Other values return LOCKS_ERR_UNSUPPORTED.
 */
#ifndef LOCKS_H_
#define LOCKS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LOCKS_ABI_VERSION 1

/* host return codes */
#define LOCKS_OK               0
#define LOCKS_ERR_INVALID_ARG (-1)   /* null pointer, bad size, k < 2, ...        */
#define LOCKS_ERR_UNSUPPORTED (-2)   /* shape outside the supported set           */
#define LOCKS_ERR_WORKSPACE   (-3)   /* workspace smaller than the size query     */
#define LOCKS_ERR_CUDA        (-4)   /* a CUDA launch failed                       */

/* device status bits, OR-ed into *status */
#define LOCKS_DEV_BAD_BLOCK_ID   0x1  /* block id < 0 or >= num_blocks: page skipped      */
#define LOCKS_DEV_WAIT_TIMEOUT   0x2  /* a bounded wait on a copy ran out: page skipped   */
#define LOCKS_DEV_NOT_CONVERGED  0x4  /* Jacobi hit max_sweeps before its tolerance       */
#define LOCKS_DEV_BAD_PAGE_ID    0x8  /* selected page id outside [0, n): entry skipped   */
#define LOCKS_DEV_BAD_SEQ_LEN    0x10 /* seq_len > max_pages * page_size: clamped         */

/* summary record element type */
#define LOCKS_SUMMARY_F32  0
#define LOCKS_SUMMARY_BF16 1
#define LOCKS_SUMMARY_I4   2   /* int4 basis, int8 coefficients and centroid */

typedef struct locks_cfg {
  int32_t batch;          /* sequences in the decode batch (>= 0)                     */
  int32_t n_q_heads;      /* query heads H_q                                           */
  int32_t n_kv_heads;     /* KV heads H_kv; H_q % H_kv == 0                            */
  int32_t head_dim;       /* d                                                         */
  int32_t page_size;      /* B, tokens per page                                        */
  int32_t rank;           /* r, modes kept per page summary                            */
  int32_t max_pages;      /* row stride of block_table (pages per sequence, at most)  */
  int32_t num_blocks;     /* physical blocks in the KV / summary pools                 */
  int32_t summary_dtype;  /* LOCKS_SUMMARY_F32, LOCKS_SUMMARY_BF16 or LOCKS_SUMMARY_I4  */
} locks_cfg_t;

/*
 * Summary record (one per (physical block, KV head)), written by
 * locks_build_summaries and read by locks_select.  Element type T is float
 * (LOCKS_SUMMARY_F32) or bf16 (LOCKS_SUMMARY_BF16).  With d = head_dim,
 * B = page_size and R = the smallest power of two >= max(rank, 4):
 *
 *   T W[R + 1][d];      W[0] = page centroid mu; W[1 + k] = basis column v_k
 *   T C[R / 4][B][4];   C[c][i][e] = coefficient c_{i, 4c + e} of token i
 *
 * Columns k >= rank and dropped (zero) modes hold zeros.  Records of one
 * KV head follow each other: record (blk, h) starts at byte
 * (blk * n_kv_heads + h) * locks_summary_record_bytes(cfg) of the pool.  The
 * basis is orthonormal (v_k^T v_l = delta_kl up to rounding), modes are in
 * descending eigenvalue order, and c_i = V^T (k_i - mu) (section 4, "Build").
 *
 * LOCKS_SUMMARY_I4 is the quantised record the paper deploys (section 4
 * "Build": the basis in int4, the coefficients and centroid in int8, with
 * per-column and per-row scales).  Each group is quantised symmetrically:
 * scale = max|x| / qmax (qmax 7 for int4, 127 for int8), code =
 * round-half-even(x / scale) clamped to [-qmax, qmax], in float32; an
 * all-zero group has scale 0.  Codes are stored biased (int4 + 8 as an
 * unsigned nibble, int8 + 128 as an unsigned byte), in the order the
 * scorer's tensor-core fragments read them.  With HDR = (R + 1) * 4 rounded
 * up to 16 bytes, KK = ceil(R / 8), and for a lane l = 4g + t (g < 8, t < 4):
 *
 *   float    vscale[R], mscale;      scale of basis column k; of the centroid
 *   uint32_t vq[R][4][4]       @HDR  word vq[k][t][j] holds, for the k-steps
 *                                    s = 2j and 2j + 1 (columns 16s + c):
 *                                    nibbles 0 / 4 = v_k at c = 2t / 2t + 1,
 *                                    nibbles 1 / 5 = c = 2t + 8 / 2t + 9 (k-step
 *                                    2j), nibbles 2 / 6 and 3 / 7 the same for
 *                                    k-step 2j + 1
 *   uint8_t  mq[32][4]         @HDR + 64R   mq[l] = mu at 16g + 2t, 16g + 2t + 1,
 *                                    16g + 2t + 8, 16g + 2t + 9
 *   uint8_t  cq[B/16][KK][32][4]  @HDR + 64R + 128   cq[m][kk][l] = c_{i,k} at
 *                                    (i, k) = (16m + g, 8kk + 2t), (16m + g,
 *                                    8kk + 2t + 1), (16m + g + 8, 8kk + 2t),
 *                                    (16m + g + 8, 8kk + 2t + 1)
 *   float    cscale[B]         @HDR + 64R + 128 + 8 B KK   scale of row c_i
 *
 * (nibble n of a word is bits 4n..4n+3; codes of columns k >= rank are 0), so
 * that v_k[x] = vscale[k] * (nibble - 8), mu[x] = mscale * (byte - 128) and
 * c_{i,k} = cscale[i] * (byte - 128).  The quantised values are those of the
 * float record's basis, coefficients and centroid.
 */
size_t locks_summary_record_bytes(const locks_cfg_t* cfg);

/* Same value as locks_summary_record_bytes (the shorter name). */
size_t locks_summary_bytes(const locks_cfg_t* cfg);

/* Bytes of workspace locks_select needs for this cfg and token budget. */
size_t locks_select_workspace_bytes(const locks_cfg_t* cfg, int32_t budget_tokens);

/* Bytes of workspace locks_sparse_decode (n_pages = its k) or
 * locks_dense_decode (n_pages = cfg->max_pages) needs. */
size_t locks_decode_workspace_bytes(const locks_cfg_t* cfg, int32_t n_pages);

/*
 * locks_build_summaries -- section 4 "Build" (and the blog review's Algorithm 1).
 *
 * For every listed block and every KV head: centre the page's B keys
 * (k_i = mu + delta_i), form the B x B Gram D D^T of the deviations, find its
 * eigenpairs with a cyclic Jacobi solver (fp32), keep the top-`rank` modes in
 * descending order (modes with sigma^2 <= 1e-5 sigma_1^2 are dropped: zero
 * basis column and coefficients), and write V = D^T U_r S_r^-1 and C = U_r S_r
 * with the centroid into the summary record.  Only complete pages (all B
 * tokens valid) may be listed.
 *
 *   k_cache      bf16 [num_blocks][n_kv_heads][B][d]
 *   block_ids    int32 [n_blocks]: physical blocks to summarise
 *   summaries    record pool, num_blocks * n_kv_heads records (see above)
 *   tail_energy  nullable float [n_blocks][n_kv_heads]: tau = sum_{k>r} sigma_k^2
 *   status       nullable int32 [n_blocks][n_kv_heads]: Jacobi sweeps used,
 *                OR-ed with LOCKS_DEV_NOT_CONVERGED << 16 / LOCKS_DEV_BAD_BLOCK_ID << 16
 *   max_sweeps   Jacobi sweep cap (>= 1; 0 selects the default, 20)
 */
int locks_build_summaries(const locks_cfg_t* cfg, const void* k_cache, const int32_t* block_ids,
                          int32_t n_blocks, void* summaries, float* tail_energy, int32_t* status,
                          int32_t max_sweeps, void* stream);

/*
 * locks_append_kv -- the cache write of one decode step, and the page
 * completions it causes (section 4 "Build": a page is summarised once, when it
 * completes; App. E (ii): one incremental build per finalised page).
 *
 * For every sequence b with t = seq_lens[b] on entry: the token's key and
 * value rows of every KV head go to slot t % B of physical block
 * block_table[b * max_pages + t / B]; seq_lens[b] becomes t + 1; and
 * completed[b] is that block when t + 1 is a multiple of B (the token
 * completed its page), else -1.  Allocating a block for a sequence's next
 * page (writing the block-table entry before the step that starts the page)
 * stays with the caller.  A sequence already holding max_pages * B tokens
 * (LOCKS_DEV_BAD_SEQ_LEN) or whose entry is not a valid block
 * (LOCKS_DEV_BAD_BLOCK_ID) is left unchanged, with completed[b] = -1.
 *
 *   k_new, v_new  bf16 [batch][n_kv_heads][d], 16-byte aligned
 *   k_cache, v_cache  the pools, 16-byte aligned; written
 *   seq_lens      int32 [batch]: read, then advanced
 *   completed     nullable int32 [batch]: written
 *   status        nullable int32[1]
 * Pass `completed` to locks_build_completed (for example on a second stream
 * that waits for this call): the page completed at step s is first a
 * selection candidate at step s + 1, so its build may overlap step s's
 * selection and decode and must finish before step s + 1's locks_select.
 */
int locks_append_kv(const locks_cfg_t* cfg, const void* k_new, const void* v_new, void* k_cache,
                    void* v_cache, const int32_t* block_table, int32_t* seq_lens,
                    int32_t* completed, int32_t* status, void* stream);

/*
 * locks_build_completed -- locks_build_summaries over a list in which an entry
 * < 0 means "no page" and is skipped without a flag (its status entries are
 * set to 0): the `completed` list that locks_append_kv writes, used as it
 * stands on the device, so no host round trip decides which pages to build.
 * Arguments as for locks_build_summaries, with block_ids = completed and
 * n_blocks = n (the batch).
 */
int locks_build_completed(const locks_cfg_t* cfg, const void* k_cache, const int32_t* completed,
                          int32_t n, void* summaries, float* tail_energy, int32_t* status,
                          int32_t max_sweeps, void* stream);

/*
 * locks_select -- section 4 "Score" (Eq. (1)), the page-mass share, the
 * share-average, and the forced-page top-(k-2) rule (section 2; Cor. 3).
 *
 * With n = ceil(seq_len / B) pages, the forced pages are {0, n-1} (page n-1 is
 * the tail, complete or not) and the candidates are the complete pages other
 * than those.  For every candidate j and query head g of the group:
 *   s_hat[g][j] = log sum_{i<B} exp((q_g^T mu_j + (V_j^T q_g)^T c_i) / sqrt(d)),
 * then m_hat_g(j) = exp(s_hat[g][j]) / sum_{j' candidate} exp(s_hat[g][j']),
 * m_bar_j = mean_g m_hat_g(j), and the selection is the forced pages plus the
 * k-2 candidates with the largest m_bar (ties: smaller page id), k = ceil(b/B).
 * If n <= k every page is selected.  Selection reads only summaries.
 *
 *   q            bf16 [batch][n_q_heads][d]
 *   summaries    record pool written by locks_build_summaries (read through block_table)
 *   block_table  int32 [batch][max_pages]
 *   seq_lens     int32 [batch]
 *   budget_tokens b >= B + 1 (k >= 2), else LOCKS_ERR_INVALID_ARG
 *   selected     int32 [batch][n_kv_heads][k]: logical page ids ascending, -1 padded
 *   page_lse     nullable float [batch][n_q_heads][max_pages]: s_hat of candidates
 *                (other entries untouched)
 *   page_share   nullable float [batch][n_kv_heads][max_pages]: m_bar of candidates
 *   workspace    >= locks_select_workspace_bytes(cfg, budget_tokens) bytes
 *   status       nullable int32[1]
 */
int locks_select(const locks_cfg_t* cfg, const void* q, const void* summaries,
                 const int32_t* block_table, const int32_t* seq_lens, int32_t budget_tokens,
                 int32_t* selected, float* page_lse, float* page_share, void* workspace,
                 size_t workspace_bytes, int32_t* status, void* stream);

/*
 * locks_sparse_decode -- attention restricted to the selected pages with the
 * softmax renormalised over them (section 2, o_S; Lemma 1), computed as
 * split-K flash decoding: each split keeps a running max, sum and weighted
 * value sum over its pages, and the splits are merged by their log-sum-exp.
 * The tail page contributes only its valid tokens.  Entries < 0 in `selected`
 * are skipped.
 *
 *   selected     int32 [batch][n_kv_heads][k] logical page ids (as locks_select writes)
 *   out          bf16 [batch][n_q_heads][d]
 *   out_lse      nullable float [batch][n_q_heads]: natural-log log-sum-exp of
 *                the scaled logits over the attended tokens (-inf if none)
 *   workspace    >= locks_decode_workspace_bytes(cfg, k) bytes
 * A sequence with no attended token gets out = 0.
 */
int locks_sparse_decode(const locks_cfg_t* cfg, const void* q, const void* k_cache,
                        const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                        const int32_t* selected, int32_t k, void* out, float* out_lse,
                        void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * locks_dense_decode -- full-cache paged decode attention (section 2, o), the
 * comparison point: the same split-K kernel over every page of each sequence.
 *   workspace    >= locks_decode_workspace_bytes(cfg, cfg->max_pages) bytes
 */
int locks_dense_decode(const locks_cfg_t* cfg, const void* q, const void* k_cache,
                       const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                       void* out, float* out_lse, void* workspace, size_t workspace_bytes,
                       int32_t* status, void* stream);

/*
 * locks_select_noalloc -- the page selection of locks_select for callers that
 * cannot allocate device memory.  The paper has no counterpart: this is a
 * packaging variant, not a step of the method.
 *
 * Callers such as a serving engine whose memory pool already owns all of the
 * GPU, a plugin whose host forbids cudaMalloc on the decode path (it can
 * synchronise the device and fragment the pool), or an embedded user without
 * an allocator get the same selection without passing a workspace: the
 * scratch lives in one fixed device array of LOCKS_SELECT_NOALLOC_MAX_BYTES
 * inside the library, which every GPU that loads the library keeps until the
 * process exits.  The call itself allocates and frees nothing.
 *
 * Arguments and outputs are those of locks_select, minus the workspace.
 * Shapes whose locks_select_workspace_bytes(cfg, budget_tokens) exceeds
 * LOCKS_SELECT_NOALLOC_MAX_BYTES are rejected with LOCKS_ERR_WORKSPACE (for
 * example, with G = 4, batch x n_kv_heads x max_pages must stay below about
 * 250,000 pages).  The array's device address is looked up by the first call
 * on a device (with that device current) and again by the first call after
 * that device's context was destroyed and re-created (cudaDeviceReset): make
 * those calls before any stream capture.  Every call clears the scratch it uses on `stream` before selecting.
 * All calls share the one array: calls that can overlap on the GPU race.
 */
#define LOCKS_SELECT_NOALLOC_MAX_BYTES (4u << 20)
int locks_select_noalloc(const locks_cfg_t* cfg, const void* q, const void* summaries,
                         const int32_t* block_table, const int32_t* seq_lens,
                         int32_t budget_tokens, int32_t* selected, float* page_lse,
                         float* page_share, int32_t* status, void* stream);

/* Static string for a LOCKS_* return code. */
const char* locks_status_string(int code);

/* LOCKS_ABI_VERSION of the loaded library. */
int locks_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LOCKS_H_ */
